"""Pins for oracle.radix (extended radix-tree matching), from the pages' rules and example."""
from oracle.radix import RadixOracle

DROP, REPOS = 1, 2


def toks(ids, pos0=0):
    return [("tok", t, pos0 + i) for i, t in enumerate(ids)]


def test_blog_history_dependence_sessions_do_not_mix():
    # [AKV-blog] section 3: both sessions share the prompt and a 4,000-token tool trace; session 1
    # drops tokens 1,000..3,500 and repositions the rest by -2,500, session 2 keeps everything.
    prefix = toks(range(4000))
    s1 = prefix + [("op", DROP, 1000, 3500, 0), ("op", REPOS, 3500, 4000, -2500)] + toks(range(7000, 7100), 1500)
    s2 = prefix + toks(range(7000, 7100), 4000)
    r = RadixOracle()
    r.insert("s1", s1)
    r.insert("s2", s2)
    # a request with session 2's history reuses session 2's state, never session 1's
    assert r.match(prefix + toks(range(7000, 7150), 4000)) == ("exact", 4100, "s2")
    # a request with session 1's history reuses session 1's
    req1 = prefix + [("op", DROP, 1000, 3500, 0), ("op", REPOS, 3500, 4000, -2500)] + toks(range(7000, 7150), 1500)
    assert r.match(req1) == ("exact", 4102, "s1")
    # a third history (a different drop) shares only the common prefix
    req3 = prefix + [("op", DROP, 0, 500, 0)] + toks(range(7000, 7010), 3500)
    kind, n, owner = r.match(req3)
    assert (kind, n) == ("exact", 4000) and owner in ("s1", "s2")


def test_retrigger_same_tokens_and_history_other_positions():
    # the same tokens and operations at positions shifted by +100: reuse after rotating every key
    path = toks(range(50)) + [("op", DROP, 10, 20, 0)] + toks(range(50, 80), 50)
    r = RadixOracle()
    r.insert("a", path)
    req = toks(range(50), 100) + [("op", DROP, 10, 20, 0)] + toks(range(50, 80), 150)
    assert r.match(req) == ("retrigger", 81, "a")
    assert r.shifts(path, req, 81) == [100] * 80


def test_tie_keeps_the_exact_match_and_strictly_longer_retrigger_wins():
    base = toks(range(20))
    r = RadixOracle()
    r.insert("exact", base + toks(range(100, 105), 20))
    r.insert("moved", toks(range(20), 7) + toks(range(100, 110), 27))
    # request equal to "exact" for 25 items; "moved" is compatible for 25 too: the tie keeps exact
    assert r.match(base + toks(range(100, 105), 20)) == ("exact", 25, "exact")
    # a request compatible with "moved" for 30 items (strictly longer) takes the retrigger match
    assert r.match(base + toks(range(100, 110), 20)) == ("retrigger", 30, "moved")


def test_walk_stops_at_the_first_token_or_operation_that_differs():
    r = RadixOracle()
    r.insert("a", toks([1, 2, 3]) + [("op", REPOS, 0, 3, 5)] + toks([4, 5], 8))
    assert r.match(toks([1, 2, 9, 4])) == ("exact", 2, "a")
    assert r.match(toks([1, 2, 3]) + [("op", REPOS, 0, 3, 6)] + toks([4, 5], 8)) == ("exact", 3, "a")
    assert r.match(toks([7, 1, 2])) == ("none", 0, None)
