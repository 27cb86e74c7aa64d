"""Sampled GPU parity at full workload sizes.

The oracle cannot hold pools of tens of GB, so it keeps only its own
bookkeeping (oracle.cache.CacheModel over every operation) plus, per token,
where its K/V came from (append key, row, original position).  Input values
come from the seeded device generator of ``runner.torch_device_kv_source`` --
torch's RNG, not this repository's kernels -- regenerated per operation when a
sample needs them.  Pool rows are read at the oracle's own (page, slot), and
the expected value of a row is the oracle's rotation of its input row.
Every token in these workloads is rotated at most once, so the expected bf16
value is round_bf16(R(pos_now - pos_append) k_input).
"""
import numpy as np
import torch

from agentic_kv_cache_gb300 import akv, build, runner, synth
from oracle import bf16, kernels, rope
from oracle.cache import CacheModel


class SampledCase:
    def __init__(self, w):
        build.build()
        self.w = w
        s = w.shape
        self.cfg = akv.config_from_shape(s, w.n_pages)
        self.pools = akv.make_pools(self.cfg)
        self.eng = akv.Engine(self.cfg, self.pools)
        self.src = runner.torch_device_kv_source(w)
        self.stream = torch.cuda.current_stream()
        self.model = CacheModel(w.n_pages, s.page_size)
        self.names = {}
        self.origin = {}  # name -> list of (key, row, position at append)

    def run(self, flush=True):
        """Replay the workload on the engine and the oracle; with `flush` the segments' sequences
        are flushed at the end (else their shifts stay pending)."""
        w, m = self.w, self.model
        for op in w.ops:
            runner.run_ops(self.eng, w, kv_source=self.src, ops=[op], names=self.names, stream=self.stream)
            kind, name = op[0], op[1]
            if kind == "alloc":
                assert m.seq_alloc() == self.names[name]
                self.origin[name] = []
            elif kind == "fork":
                assert m.seq_fork(self.names[op[2]], op[3]) == self.names[name]
                self.origin[name] = self.origin[op[2]][:op[3]]
            elif kind == "append":
                sid = self.names[name]
                m.append(sid, op[2])
                pos = m.state(sid)["pos"][-op[2]:] if op[2] else []
                self.origin[name] += [(op[3], i, pos[i]) for i in range(op[2])]
            elif kind == "drop":
                m.drop(self.names[name], op[2], op[3])
            elif kind == "repos":
                m.repos(self.names[name], op[2], op[3], op[4])
            elif kind == "splice":
                sid = self.names[name]
                m.splice(sid, op[2], op[3], op[4])
                pos = m.state(sid)["pos"][op[2]:op[2] + op[4]]
                self.origin[name] = (self.origin[name][:op[2]] + [(op[5], i, pos[i]) for i in range(op[4])]
                                     + self.origin[name][op[3]:])
            elif kind == "flush":
                m.flush([self.names[name]])
        if flush:
            ids = sorted({self.names[g["seq"]] for g in w.segments})
            m.flush(ids)
            for i in ids:
                self.eng.flush(i, stream=self.stream)
        torch.cuda.synchronize()
        assert self.eng.check_device_error(self.stream) == 0

    def compact(self, name):
        """Compact `name` on the engine and in the oracle (pending shifts fused into the copy); the
        dropped tokens leave the logical sequence, so the sample origins follow.  Returns the
        oracle's copy list."""
        sid = self.names[name]
        vis = [t.vis for t in self.model.seqs[sid]]
        copies = self.model.compact(sid)
        self.eng.compact(sid, stream=self.stream)
        torch.cuda.synchronize()
        assert self.eng.check_device_error(self.stream) == 0
        assert self.eng.fragmentation(sid) == self.model.fragmentation(sid)
        self.origin[name] = [o for o, v in zip(self.origin[name], vis) if v]
        return copies

    # ------------------------------------------------------------- inputs
    def inputs(self, refs, layer=None):
        """Input rows for a list of (key, row): (K, V) float64 arrays [n][L][H][d] (or [n][H][d] for one layer)."""
        n_of = {}
        for op in self.w.ops:
            if op[0] == "append":
                n_of[op[3]] = op[2]
            elif op[0] == "splice":
                n_of[op[5]] = op[4]
        s = self.w.shape
        lead = () if layer is not None else (s.n_layers,)
        K = np.empty((len(refs),) + lead + (s.n_kv_heads, s.d_rot))
        V = np.empty((len(refs),) + lead + (s.n_kv_heads, s.d_v))
        by_key = {}
        for j, (key, row) in enumerate(refs):
            by_key.setdefault(key, []).append((j, row))
        for key, items in by_key.items():
            k, v = self.src(key, n_of[key])
            if layer is not None:
                k, v = k[layer], v[layer]          # [n][H][d]
            else:
                k, v = k.transpose(0, 1), v.transpose(0, 1)  # [n][L][H][d]
            idx = torch.tensor([r for _, r in items], device=k.device)
            pos = np.array([j for j, _ in items])
            K[pos] = k[idx].double().cpu().numpy()
            V[pos] = v[idx].double().cpu().numpy()
            del k, v
        torch.cuda.empty_cache()
        return K, V

    def expected(self, name, idxs, layer=None):
        """Oracle K (rotated once by pos_now - pos_append, rounded) and V of tokens idxs of `name`."""
        s = self.w.shape
        refs = [self.origin[name][i][:2] for i in idxs]
        K_in, V = self.inputs(refs, layer)
        toks = self.model.seqs[self.names[name]]
        d = np.array([toks[i].pos - self.origin[name][i][2] for i in idxs], np.float64)
        K = K_in.copy()
        moved = d != 0
        if moved.any():
            km = K_in[moved]
            dm = np.broadcast_to(d[moved].reshape((-1,) + (1,) * (km.ndim - 2)), km.shape[:-1])
            K[moved] = bf16.round_bf16(rope.repos(km, dm, s.rope_base, s.rope_layout))
        return K_in, K, V, moved

    # ------------------------------------------------------------- checks
    def check_repos(self, n_samples, rng):
        """Sampled tokens of every live sequence: GPU K rows (all layers, heads) vs the oracle."""
        s = self.w.shape
        names = [n for n in self.origin if self.names[n] in self.model.seqs]
        worst, n_eq, n_all, n_rot = 0.0, 0, 0, 0
        for name in names:
            toks = self.model.seqs[self.names[name]]
            idxs = sorted(set(int(x) for x in rng.integers(0, len(toks), size=max(1, n_samples // len(names)))))
            K_in, want, _, moved = self.expected(name, idxs)
            kp = torch.tensor([toks[i].kp for i in idxs], device="cuda")
            sl = torch.tensor([toks[i].slot for i in idxs], device="cuda")
            got = self.pools[0][:, kp, :, sl, :].double().cpu().numpy()  # [n][L][H][d]: index dims first
            assert np.array_equal(got[~moved], want[~moved]), name
            if not moved.any():
                continue
            g, wv, xin = got[moved], want[moved], K_in[moved]
            a, b = rope.pair_indices(s.d_rot, s.rope_layout)
            term = np.empty_like(xin)
            t = 2.0 ** -20 * (np.abs(xin[..., a]) + np.abs(xin[..., b]))
            term[..., a] = t
            term[..., b] = t
            r = np.abs(g - wv) / (bf16.ulp_bf16(wv) + term)
            worst = max(worst, float(r.max()))
            n_eq += int((g == wv).sum())
            n_all += g.size
            n_rot += int(moved.sum())
        assert worst <= 1.0, worst
        if n_all:
            assert n_eq / n_all >= 0.999, n_eq / n_all
        return n_rot, worst

    def check_values(self, n_samples, rng):
        """Sampled tokens of every live sequence: GPU V rows (all layers, heads) bit-identical to
        the appended values."""
        names = [n for n in self.origin if self.names[n] in self.model.seqs]
        n_checked = 0
        for name in names:
            toks = self.model.seqs[self.names[name]]
            idxs = sorted(set(int(x) for x in rng.integers(0, len(toks), size=max(1, n_samples // len(names)))))
            _, _, want, _ = self.expected(name, idxs)
            vp = torch.tensor([toks[i].vp for i in idxs], device="cuda")
            sl = torch.tensor([toks[i].slot for i in idxs], device="cuda")
            got = self.pools[1][:, vp, :, sl, :].double().cpu().numpy()  # [n][L][H][d]
            assert np.array_equal(got, want), name
            n_checked += len(idxs)
        return n_checked

    def sample_rows(self, q_len, n_random, rng):
        """Query rows to check in one segment: the first and last row of every 128-row query tile
        (a tile holds 128 / G tokens of one kv group, G = query heads per kv head), so every
        work item of the launch over the segment -- split across CTAs or not -- has checked
        rows, plus n_random further rows drawn without replacement."""
        s = self.w.shape
        per_tile = 128 // (s.n_q_heads // s.n_kv_heads)
        starts = np.arange(0, q_len, per_tile)
        edge = np.concatenate([starts, np.minimum(starts + per_tile, q_len) - 1])
        rest = np.setdiff1d(np.arange(q_len), edge)
        pick = rng.choice(rest, size=min(n_random, rest.size), replace=False)
        return np.unique(np.concatenate([edge, pick]))

    def check_attention(self, layer, rows_per_segment, rng, segments=None):
        """Sampled query rows of the given segments (see sample_rows): GPU output vs the float64
        oracle, every row against the segment's full visible list.  The oracle is evaluated one
        query head at a time in a thread pool (numpy releases the GIL in its kernels)."""
        import os
        from concurrent.futures import ThreadPoolExecutor
        from oracle import attention
        s, w = self.w.shape, self.w
        q32 = synth.q_array(w, layer)
        nq = q32.shape[0]
        qd = torch.from_numpy(q32).cuda().to(torch.bfloat16)
        o = torch.full((nq, s.n_q_heads, s.d_v), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((nq, s.n_q_heads), dtype=torch.float32, device="cuda")
        self.eng.attend(layer, runner.engine_segments(w, self.names), qd, nq, o, lse, s.scale, stream=self.stream)
        torch.cuda.synchronize()
        assert self.eng.check_device_error(self.stream) == 0
        segs = range(len(w.segments)) if segments is None else segments
        group = s.n_q_heads // s.n_kv_heads
        n_threads = max(1, min(16, os.cpu_count() or 1))
        worst, n_rows = 0.0, 0
        for si in segs:
            g = w.segments[si]
            name = g["seq"]
            runs, kv_len = self.model.segment_runs(self.names[name], g["kv_end"], g["q_len"], g["hide"])
            # visible entries in logical order, with their token indices
            hidden = np.zeros(g["kv_end"], bool)
            for a, b in g["hide"]:
                hidden[a:b] = True
            toks = self.model.seqs[self.names[name]]
            vis = [i for i in range(g["kv_end"]) if toks[i].vis and not hidden[i]]
            assert len(vis) == kv_len
            _, K, V, _ = self.expected(name, vis, layer)   # [kv][H][d]
            if s.mla:
                K = np.concatenate([V, K], axis=-1)
            rows = self.sample_rows(g["q_len"], rows_per_segment, rng)
            qb = bf16.round_bf16(q32[g["q_row0"]:g["q_row0"] + g["q_len"]].astype(np.float64))

            def one_head(h):
                kv = h // group
                return attention.segment_attention(qb[:, h:h + 1], K[:, kv:kv + 1], V[:, kv:kv + 1], s.scale,
                                                   rows=rows)

            with ThreadPoolExecutor(n_threads) as ex:
                parts = list(ex.map(one_head, range(s.n_q_heads)))
            want_o = np.concatenate([p[0] for p in parts], axis=1)
            want_lse = np.concatenate([p[1] for p in parts], axis=1)
            idx = g["q_row0"] + torch.from_numpy(rows).cuda()
            got_o = o[idx].double().cpu().numpy()
            got_lse = lse[idx].double().cpu().numpy()
            err = float(np.abs(got_o - want_o).max())
            worst = max(worst, err)
            assert err <= 2e-2, (si, err)
            assert np.abs(got_lse - want_lse).max() <= 2e-2
            n_rows += len(rows)
        return worst, n_rows
