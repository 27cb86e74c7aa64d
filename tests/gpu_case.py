"""GPU parity harness: one workload run through the engine (device pools) and
through the oracle (its own bookkeeping and its own float32-held bf16 pools,
built from the same seeded synth values, never from the GPU's output)."""
import numpy as np
import torch

from agentic_kv_cache_gb300 import akv, build, runner, synth
from oracle import attention, bf16, kernels
from oracle.cache import CacheModel


def bf16_of(x32):
    """The bf16 values (held in float32) of a float32 array, rounded by the oracle."""
    return bf16.round_bf16(np.asarray(x32, np.float64)).astype(np.float32)


class Case:
    def __init__(self, w, device_values=False):
        build.build()
        self.w = w
        s = w.shape
        self.cfg = akv.config_from_shape(s, w.n_pages)
        self.pools = akv.make_pools(self.cfg)
        self.eng = akv.Engine(self.cfg, self.pools)
        self.model = CacheModel(w.n_pages, s.page_size)
        L, P, H, S = s.n_layers, w.n_pages, s.n_kv_heads, s.page_size
        self.kp = np.zeros((L, P, H, S, s.d_rot), np.float32)
        # per rotated element: the float32 rounding allowance of the rotation,
        # 2^-20 * (|x_a| + |x_b|) of its input pair (see compare_rotated)
        self.kterm = np.zeros((L, P, H, S, s.d_rot), np.float32)
        self.vp = np.zeros((L, P, H, S, s.d_v), np.float32)
        self.stream = torch.cuda.current_stream()
        self.names_e = {}
        self.names_o = {}
        self.flush_runs = []

    # ----------------------------------------------------------- replay
    def _values(self, key, n):
        k32, v32 = synth.kv_arrays(self.w, key, n)
        return k32, v32

    def run_ops(self, ops=None):
        w = self.w
        for op in (w.ops if ops is None else ops):
            kind = op[0]
            if kind in ("append", "splice"):
                n, key = (op[2], op[3]) if kind == "append" else (op[4], op[5])
                k32, v32 = self._values(key, n)
                kd = torch.from_numpy(k32).cuda().to(torch.bfloat16)
                vd = torch.from_numpy(v32).cuda().to(torch.bfloat16)
                runner.run_ops(self.eng, w, kv_source=lambda *_: (kd, vd), ops=[op], names=self.names_e)
                seq = self.names_o[op[1]]
                slots = (self.model.append(seq, n) if kind == "append"
                         else self.model.splice(seq, op[2], op[3], op[4]))
                kb, vb = bf16_of(k32), bf16_of(v32)
                for i, (kp, vp, sl) in enumerate(slots):
                    self.kp[:, kp, :, sl, :] = kb[:, i]
                    self.vp[:, vp, :, sl, :] = vb[:, i]
            else:
                runner.run_ops(self.eng, w, ops=[op], names=self.names_e, stream=self.stream)
                if kind == "alloc":
                    self.names_o[op[1]] = self.model.seq_alloc()
                elif kind == "fork":
                    self.names_o[op[1]] = self.model.seq_fork(self.names_o[op[2]], op[3])
                elif kind == "drop":
                    self.model.drop(self.names_o[op[1]], op[2], op[3])
                elif kind == "repos":
                    self.model.repos(self.names_o[op[1]], op[2], op[3], op[4])
                elif kind == "flush":
                    runs = self.model.flush([self.names_o[op[1]]])
                    self._apply_runs(runs)
        assert self.names_e == self.names_o

    def _apply_runs(self, runs):
        s = self.w.shape
        from oracle import rope
        for src, dst, lo, hi, d in runs:
            x = np.abs(self.kp[:, src, :, lo:hi, :].astype(np.float64))
            a, b = rope.pair_indices(s.d_rot, s.rope_layout)
            t = 2.0 ** -20 * (x[..., a] + x[..., b])
            view = self.kterm[:, dst, :, lo:hi, :]
            view[..., a] = t
            view[..., b] = t
        kernels.repos_runs(self.kp, runs, s.rope_base, s.rope_layout, out=self.kp)
        self.flush_runs.extend(runs)

    def flush_segments(self, engine=True):
        """The flush attention performs: every segment's sequence, increasing id.  With
        engine=False only the oracle materialises (the fused path leaves the GPU pools as they are)."""
        ids = sorted({self.names_o[g["seq"]] for g in self.w.segments})
        runs = self.model.flush(ids)
        self._apply_runs(runs)
        if engine:
            for i in ids:
                self.eng.flush(i, stream=self.stream)
        return runs

    # ------------------------------------------------------------ pools
    def gpu_pools(self):
        torch.cuda.synchronize()
        return (self.pools[0].float().cpu().numpy(), self.pools[1].float().cpu().numpy())

    # -------------------------------------------------------- attention
    def queries(self, layer=0):
        q32 = synth.q_array(self.w, layer)
        return q32, torch.from_numpy(q32).cuda().to(torch.bfloat16)

    def attend_gpu(self, layer=0, with_lse=True, fused=False):
        s = self.w.shape
        q32, qd = self.queries(layer)
        nq = q32.shape[0]
        o = torch.full((nq, s.n_q_heads, s.d_v), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((nq, s.n_q_heads), float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
        segs = runner.engine_segments(self.w, self.names_e)
        self.eng.attend(layer, segs, qd, nq, o, lse, s.scale, stream=self.stream, fused=fused)
        torch.cuda.synchronize()
        assert self.eng.check_device_error(self.stream) == 0
        return q32, o.float().cpu().numpy(), (lse.cpu().numpy() if with_lse else None)

    def attend_oracle(self, q32, seg_index, rows, layer=0):
        """Oracle output of one segment for selected query rows (indices inside the segment)."""
        s = self.w.shape
        g = self.w.segments[seg_index]
        runs, kv_len = self.model.segment_runs(self.names_o[g["seq"]], g["kv_end"], g["q_len"], g["hide"])
        qb = bf16_of(q32[g["q_row0"]:g["q_row0"] + g["q_len"]])
        return kernels.attend_segment(qb, self.kp, self.vp, layer, runs, s.scale, mla=s.mla, rows=rows)
