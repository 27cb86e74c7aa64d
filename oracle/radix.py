"""Extended radix-tree matching by brute force (test infrastructure only).

[AKV-blog] section 3 "Resolving History Dependence via Extended Radix Trees":
an edge carries the token sequence and the ordered cache operations applied
to it; a lookup walks tokens and verifies the operation history, and when the
tokens match but the history diverges the state branches.  [AKV-notes]
"Cache Reuse Matching Rules": every cached token is T(x, p), token x whose
cached key encodes position p;

* exact match: same tokens, same positions, identical operation record along
  the path -> reuse the cache as it is;
* retrigger match: same tokens and identical operation history, positions may
  differ -> reuse after rotating the keys (the hidden states are the same);
* lookup: the longest exact-match prefix first, then from the root the
  history-compatible branch, which replaces it only if strictly longer (a
  tie keeps the exact match); a walk stops at the first token or operation
  that differs.

A path is a list of items: ("tok", x, p) for a cached token, or ("op", code,
a, b, c) for a cache operation applied at that point.  The oracle keeps every
inserted path and compares the request against each one; ties between paths
of equal match length go to the earliest inserted.
"""


def _exact_len(path, req):
    n = 0
    for a, b in zip(path, req):
        if a != b:
            break
        n += 1
    return n


def _key(item):
    """The item without the position of a token (what a retrigger match compares)."""
    return item[:2] if item[0] == "tok" else item


def _compat_len(path, req):
    n = 0
    for a, b in zip(path, req):
        if _key(a) != _key(b):
            break
        n += 1
    return n


class RadixOracle:
    def __init__(self):
        self.paths = []  # (owner, items), insertion order

    def insert(self, owner, items):
        self.paths.append((owner, [tuple(x) for x in items]))

    def match(self, req):
        """(kind, n_items, owner): kind "exact", "retrigger" or "none"."""
        req = [tuple(x) for x in req]
        best_e = (0, None)
        best_r = (0, None)
        for owner, path in self.paths:
            e = _exact_len(path, req)
            if e > best_e[0]:
                best_e = (e, owner)
            r = _compat_len(path, req)
            if r > best_r[0]:
                best_r = (r, owner)
        if best_r[0] > best_e[0]:
            return "retrigger", best_r[0], best_r[1]
        if best_e[0] > 0:
            return "exact", best_e[0], best_e[1]
        return "none", 0, None

    @staticmethod
    def shifts(path, req, n_items):
        """Per token of the first n_items: request position - cached position."""
        out = []
        for a, b in zip(path[:n_items], req[:n_items]):
            if a[0] == "tok":
                out.append(b[2] - a[2])
        return out
