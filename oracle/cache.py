"""Paged KV-cache bookkeeping model (test infrastructure only).

This is the oracle's own statement of the append / drop / repos contract and
of Leyline's AMORTIZE splice over a paged cache.  It produces the page map,
per-token positions, the run list a flush must rotate and the run list a
segment attends over; the engine has to reproduce every one of them bit for bit.

Sources:

* [AKV-notes] section 1 "Problem & Solution": the three cache operations
  append / drop / repos, interleaved by the harness.
* [AKV-blog] section 2 "The Drop Primitive": drop marks a span invisible to
  attention and does not deallocate; the paged kernel skips those entries.
* [AKV-blog] section 2 "The Repos Primitive ...": repos re-rotates retained
  keys by Delta; [Leyline] "Method": several non-overlapping directives compose
  into one rotation per token, Delta of either sign.
* [AKV-notes] section 2 "Motivation": the position index is kept apart from the
  logical index and from the cache size.
* [AKV-notes] section 3 "Cache Management": reuse after repos copies the
  cache state and rotates the copy (a new branch); [AKV-blog] section 3: forks
  share physical blocks through copy-on-write page references.
* [Leyline] "Method": splice D = (s_start, s_end, R) replaces a span by a stub
  R; every later slot shifts by Delta = |R| - (s_end - s_start); only the
  position-encoded key part is rotated, K_nope and V are untouched.
* [AKV-notes] section 3 "Segment-Batch Attention": queries are partitioned
  into segments by visible history; each segment selects its KV pages and runs
  standard causal attention, with no dense mask.

Rules where the pages are silent (the engine implements the same rules):

* Two page pools of the same size, one for the rotated key part ("K": all of K
  under GQA, K_pe under MLA) and one for the rest ("V": V under GQA, the latent
  under MLA).  Each has its own reference counts; a fresh page is always the
  lowest free id of its pool.
* refcount(p) = number of live sequences having at least one token in page p.
* append fills the page of the logically last token at slot+1 when that
  token's K page and V page both have refcount 1 and the page has room;
  otherwise it opens new pages (one K page and one V page at a time).
  Default positions continue from the last token's position + 1 (0 if empty).
* drop never frees memory.  repos only records a pending Delta per token.
* flush materialises pending Delta of *visible* tokens only (dropped tokens
  are never read again, so they keep theirs pending).  A K page with refcount
  1 is rotated in place; a shared one is copied (copy-on-write of the K page
  only, the V page stays shared) together with every visible token of the
  sequence in it, rotated or not.
* splice removes tokens [s, e) from the logical sequence (pages that the
  sequence no longer references are released), writes the stub into fresh
  pages, inserts it at logical index s, and adds Delta = n_stub - (e - s) to
  the pending Delta of every later token.  Stub positions default to the
  position of token s (or last + 1), counting up.
* Positions are int32; an operation that would leave int32 fails.
* Every failing operation leaves the state unchanged.
* Compaction ([AKV-blog] "Dilemma 2: Memory Fragmentation in Paged Pools":
  surviving blocks are copied into contiguous physical spans).  The
  fragmentation of a sequence is the share of the slots of its K pages that do
  not hold one of its visible tokens: 1 - n_visible / (n_K_pages * page).
  compact(seq) writes the visible tokens, in logical order, densely into fresh
  pages (lowest free ids, one K and one V page per `page` tokens, slot =
  index mod page), with any pending Delta applied to the copied key (so the
  copy has Delta 0 and position pos + Delta), the value copied unchanged.
  Dropped tokens leave the logical sequence (nothing can read them again), so
  later logical indices move down, as after a splice.  The old pages lose the
  sequence's reference.  New pages are taken before old ones are released, so
  the pools must hold ceil(n_visible / page) free pages each.
"""
import heapq

INT32_MIN = -(2 ** 31)
INT32_MAX = 2 ** 31 - 1


class CacheError(Exception):
    """An operation was rejected; ``code`` names the status the engine returns."""

    def __init__(self, code, msg):
        super().__init__(f"{code}: {msg}")
        self.code = code


class Tok:
    __slots__ = ("kp", "vp", "slot", "pos", "delta", "vis")

    def __init__(self, kp, vp, slot, pos, delta=0, vis=True):
        self.kp, self.vp, self.slot = kp, vp, slot
        self.pos, self.delta, self.vis = pos, delta, vis

    def copy(self):
        return Tok(self.kp, self.vp, self.slot, self.pos, self.delta, self.vis)

    @property
    def eff(self):
        """The position the token has once its pending Delta is applied."""
        return self.pos + self.delta


class _Pool:
    """Reference counts of one page pool, lowest-free-id-first allocation."""

    def __init__(self, n):
        self.rc = [0] * n
        self.free = list(range(n))  # a valid min-heap
        self.n_free = n

    def alloc(self):
        p = heapq.heappop(self.free)
        assert self.rc[p] == 0
        self.rc[p] = 1
        self.n_free -= 1
        return p

    def inc(self, p):
        self.rc[p] += 1

    def dec(self, p):
        self.rc[p] -= 1
        assert self.rc[p] >= 0
        if self.rc[p] == 0:
            heapq.heappush(self.free, p)
            self.n_free += 1


def _check_i32(v, what):
    if not (INT32_MIN <= v <= INT32_MAX):
        raise CacheError("OVERFLOW", f"{what} {v} leaves int32")


class CacheModel:
    def __init__(self, n_pages, page_size):
        if n_pages <= 0 or page_size <= 0:
            raise CacheError("ARG", "pool sizes must be positive")
        self.n_pages, self.page = n_pages, page_size
        self.K, self.V = _Pool(n_pages), _Pool(n_pages)
        self.seqs = {}
        self._free_ids = []
        self._next_id = 0

    # ---------------------------------------------------------------- helpers
    def _seq(self, seq):
        if seq not in self.seqs:
            raise CacheError("ARG", f"sequence {seq} is not live")
        return self.seqs[seq]

    @staticmethod
    def _pages(toks):
        return {t.kp for t in toks}, {t.vp for t in toks}

    def _new_id(self):
        if self._free_ids:
            return heapq.heappop(self._free_ids)
        self._next_id += 1
        return self._next_id - 1

    @staticmethod
    def _next_pos(toks):
        return toks[-1].eff + 1 if toks else 0

    # ------------------------------------------------------------- operations
    def seq_alloc(self):
        sid = self._new_id()
        self.seqs[sid] = []
        return sid

    def seq_fork(self, src, n_prefix):
        """New sequence sharing tokens [0, n_prefix) of src (refcounts, no copy)."""
        toks = self._seq(src)
        if not (0 <= n_prefix <= len(toks)):
            raise CacheError("RANGE", "fork prefix outside the sequence")
        child = [t.copy() for t in toks[:n_prefix]]
        kps, vps = self._pages(child)
        for p in kps:
            self.K.inc(p)
        for p in vps:
            self.V.inc(p)
        sid = self._new_id()
        self.seqs[sid] = child
        return sid

    def seq_free(self, seq):
        toks = self._seq(seq)
        kps, vps = self._pages(toks)
        for p in kps:
            self.K.dec(p)
        for p in vps:
            self.V.dec(p)
        del self.seqs[seq]
        heapq.heappush(self._free_ids, seq)

    def append(self, seq, n, pos=None):
        """Append n tokens; returns [(k_page, v_page, slot)] for each new token."""
        toks = self._seq(seq)
        if n < 0:
            raise CacheError("ARG", "negative token count")
        if pos is None:
            start = self._next_pos(toks)
            if n:
                _check_i32(start + n - 1, "position")
            pos = [start + i for i in range(n)]
        else:
            pos = [int(p) for p in pos]
            if len(pos) != n:
                raise CacheError("ARG", "position count differs from n")
            for p in pos:
                _check_i32(p, "position")
        room, kp, vp, slot = 0, -1, -1, -1
        if toks:
            last = toks[-1]
            if self.K.rc[last.kp] == 1 and self.V.rc[last.vp] == 1:
                room = self.page - 1 - last.slot
                kp, vp, slot = last.kp, last.vp, last.slot
        need = 0 if n <= room else -(-(n - room) // self.page)
        if need > self.K.n_free or need > self.V.n_free:
            raise CacheError("NO_PAGES", f"append needs {need} pages")
        out = []
        for i in range(n):
            if room > 0:
                slot += 1
                room -= 1
            else:
                kp, vp, slot = self.K.alloc(), self.V.alloc(), 0
                room = self.page - 1
            toks.append(Tok(kp, vp, slot, pos[i]))
            out.append((kp, vp, slot))
        return out

    def drop(self, seq, s, e):
        toks = self._seq(seq)
        if not (0 <= s <= e <= len(toks)):
            raise CacheError("RANGE", "drop span outside the sequence")
        for t in toks[s:e]:
            t.vis = False

    def repos(self, seq, s, e, delta):
        toks = self._seq(seq)
        if not (0 <= s <= e <= len(toks)):
            raise CacheError("RANGE", "repos span outside the sequence")
        _check_i32(delta, "delta")
        for t in toks[s:e]:
            _check_i32(t.delta + delta, "composed delta")
            _check_i32(t.eff + delta, "position")
        for t in toks[s:e]:
            t.delta += delta

    def splice(self, seq, s, e, n_stub, pos=None):
        """AMORTIZE splice; returns [(k_page, v_page, slot)] for the stub tokens."""
        toks = self._seq(seq)
        if not (0 <= s <= e <= len(toks)) or n_stub < 0:
            raise CacheError("RANGE", "splice span outside the sequence")
        delta = n_stub - (e - s)
        _check_i32(delta, "delta")
        if pos is None:
            p0 = toks[s].eff if s < len(toks) else self._next_pos(toks)
            if n_stub:
                _check_i32(p0 + n_stub - 1, "position")
            pos = [p0 + i for i in range(n_stub)]
        else:
            pos = [int(p) for p in pos]
            if len(pos) != n_stub:
                raise CacheError("ARG", "position count differs from n_stub")
            for p in pos:
                _check_i32(p, "position")
        for t in toks[e:]:
            _check_i32(t.delta + delta, "composed delta")
            _check_i32(t.eff + delta, "position")
        keep = toks[:s] + toks[e:]
        k_before, v_before = self._pages(toks)
        k_after, v_after = self._pages(keep)
        k_rel, v_rel = k_before - k_after, v_before - v_after
        need = -(-n_stub // self.page)
        k_free = self.K.n_free + sum(1 for p in k_rel if self.K.rc[p] == 1)
        v_free = self.V.n_free + sum(1 for p in v_rel if self.V.rc[p] == 1)
        if need > k_free or need > v_free:
            raise CacheError("NO_PAGES", f"splice needs {need} pages")
        for p in k_rel:
            self.K.dec(p)
        for p in v_rel:
            self.V.dec(p)
        stub, out = [], []
        kp = vp = -1
        for i in range(n_stub):
            if i % self.page == 0:
                kp, vp = self.K.alloc(), self.V.alloc()
            stub.append(Tok(kp, vp, i % self.page, pos[i]))
            out.append((kp, vp, i % self.page))
        for t in toks[e:]:
            t.delta += delta
        toks[:] = toks[:s] + stub + toks[e:]
        return out

    # ------------------------------------------------------------------ flush
    def _flush_plan(self, toks, rc):
        """Pages of the visible moving tokens (first-appearance order) and which need a copy."""
        order = []
        seen = set()
        for t in toks:
            if t.vis and t.delta != 0 and t.kp not in seen:
                seen.add(t.kp)
                order.append(t.kp)
        return order, [p for p in order if rc[p] > 1]

    def flush(self, seqs=None):
        """Materialise pending Delta; returns the run list [(src, dst, lo, hi, delta)].

        seqs: iterable of sequence ids, or None for every live sequence; they
        are processed in increasing id order.
        """
        ids = sorted(self.seqs) if seqs is None else sorted(set(seqs))
        for sid in ids:
            self._seq(sid)
        # Check the page budget first so that a failure changes nothing.
        rc = list(self.K.rc)
        need = 0
        for sid in ids:
            toks = self.seqs[sid]
            _, cow = self._flush_plan(toks, rc)
            need += len(cow)
            # The sequence leaves a copied page entirely unless one of its
            # dropped tokens stays behind in it; then the page loses a reference.
            for p in cow:
                if not any(t.kp == p and not t.vis for t in toks):
                    rc[p] -= 1
        if need > self.K.n_free:
            raise CacheError("NO_PAGES", f"flush needs {need} copy-on-write pages")
        runs = []
        for sid in ids:
            runs.extend(self._flush_seq(self.seqs[sid]))
        return runs

    def _flush_seq(self, toks):
        order, cow = self._flush_plan(toks, self.K.rc)
        if not order:
            return []
        dst = {p: p for p in order}
        for p in cow:
            dst[p] = self.K.alloc()
        # Which tokens this flush writes: visible tokens whose page moves
        # (copied, rotated or not) and visible tokens with a pending Delta.
        moved = set(cow)
        emit = [t.vis and (t.delta != 0 or t.kp in moved) for t in toks]
        runs = []
        cur = None
        for t, em in zip(toks, emit):
            if not em:
                cur = None
                continue
            key = (t.kp, dst[t.kp] if t.kp in dst else t.kp, t.delta)
            if cur is not None and cur[0] == key and t.slot == cur[2]:
                cur[2] += 1
            else:
                cur = [key, t.slot, t.slot + 1]
                runs.append(cur)
        out = [(k[0], k[1], lo, hi, k[2]) for k, lo, hi in runs]
        for t, em in zip(toks, emit):
            if em:
                if t.kp in moved:
                    t.kp = dst[t.kp]
                t.pos += t.delta
                t.delta = 0
        for p in cow:  # drop the reference when no (dropped) token stays behind
            if not any(t.kp == p for t in toks):
                self.K.dec(p)
        return out

    # -------------------------------------------------------------- segments
    def segment_runs(self, seq, kv_end, q_len, hide=()):
        """Run list [(k_page, v_page, lo, hi)] and kv_len of one attention segment.

        The segment sees the visible tokens of [0, kv_end) outside the hidden
        spans, in logical order; its queries are tokens [kv_end - q_len, kv_end),
        which must be the last q_len of those entries.
        """
        toks = self._seq(seq)
        if not (1 <= q_len <= kv_end <= len(toks)):
            raise CacheError("RANGE", "segment outside the sequence")
        hidden = [False] * kv_end
        for a, b in hide:
            if not (0 <= a <= b <= kv_end):
                raise CacheError("RANGE", "hidden span outside the segment")
            for i in range(a, b):
                hidden[i] = True
        for i in range(kv_end - q_len, kv_end):
            if not toks[i].vis or hidden[i]:
                raise CacheError("ARG", "a query token of the segment is not visible")
        runs = []
        cur = None
        n = 0
        for i in range(kv_end):
            t = toks[i]
            if not t.vis or hidden[i]:
                continue
            if t.delta != 0:
                raise CacheError("ARG", "segment reads a token with a pending delta")
            n += 1
            if cur is not None and cur[0] == t.kp and cur[1] == t.vp and t.slot == cur[3]:
                cur[3] += 1
            else:
                cur = [t.kp, t.vp, t.slot, t.slot + 1]
                runs.append(cur)
        return [tuple(r) for r in runs], n

    # -------------------------------------------------------------- compaction
    def fragmentation(self, seq):
        """1 - visible tokens / slots of the sequence's K pages (0.0 for an empty sequence)."""
        toks = self._seq(seq)
        kps, _ = self._pages(toks)
        if not kps:
            return 0.0
        return 1.0 - sum(1 for t in toks if t.vis) / (len(kps) * self.page)

    def compact(self, seq):
        """Copy the visible tokens densely into fresh pages; returns the copy list
        [(src_k, src_v, src_slot, dst_k, dst_v, dst_slot, delta)], one entry per kept token."""
        toks = self._seq(seq)
        keep = [t for t in toks if t.vis]
        need = -(-len(keep) // self.page)
        if need > self.K.n_free or need > self.V.n_free:
            raise CacheError("NO_PAGES", f"compaction needs {need} pages")
        kps, vps = self._pages(toks)
        out, new = [], []
        kp = vp = -1
        for i, t in enumerate(keep):
            if i % self.page == 0:
                kp, vp = self.K.alloc(), self.V.alloc()
            out.append((t.kp, t.vp, t.slot, kp, vp, i % self.page, t.delta))
            new.append(Tok(kp, vp, i % self.page, t.pos + t.delta))
        for p in kps:
            self.K.dec(p)
        for p in vps:
            self.V.dec(p)
        toks[:] = new
        return out

    # ---------------------------------------------------------------- export
    def state(self, seq):
        """Per-token arrays (k_page, v_page, slot, pos, delta, visible) of one sequence."""
        toks = self._seq(seq)
        return {
            "k_page": [t.kp for t in toks],
            "v_page": [t.vp for t in toks],
            "slot": [t.slot for t in toks],
            "pos": [t.pos for t in toks],
            "delta": [t.delta for t in toks],
            "visible": [int(t.vis) for t in toks],
        }

    def refcounts(self):
        return list(self.K.rc), list(self.V.rc)
