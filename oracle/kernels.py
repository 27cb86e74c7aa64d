"""What the two GPU kernels compute, over paged pools (test infrastructure only).

The pools follow the engine's layout: a rotated-key pool ``kpool`` of shape
[L][P][H][page][d_rot] (all of K under GQA; K_pe with H = 1 under MLA) and an
unrotated pool ``vpool`` [L][P][H][page][d_v] (V under GQA; the latent under
MLA, which serves as K_nope and as V).  Values are float64 holding exact
bfloat16 numbers.

repos: [AKV-blog] section 2 "The Repos Primitive ..." and [Leyline] "Method":
each retained key row is rotated once by its composed Delta, k' = R(Delta) k,
and stored back as bfloat16.  Under MLA only K_pe rotates.

attend: [AKV-notes] section 3 "Segment-Batch Attention": gather the segment's
KV entries through its run list, then causal attention (oracle.attention).
"""
import numpy as np

from . import attention, bf16, rope


def repos_runs(kpool, runs, base, layout="interleaved", out=None):
    """Apply a flush run list [(src, dst, lo, hi, delta)] to a copy of kpool.

    Every run reads rows [lo, hi) of page src in every layer and head, rotates
    them by delta in float64, rounds to bfloat16 and writes them to the same
    rows of page dst.  Runs are applied one after another in list order.
    Without ``out`` every run reads the pool as it was before the flush.  With
    ``out=kpool`` the pool is updated in place and a run reads what earlier
    runs left: a flush of two sequences sharing a page lists the copy of that
    page (copy-on-write for the first sharer) before the in-place rotation of
    the same page (for the last sharer), so the copy reads the unrotated rows
    and the result equals the out-of-place one.  No two runs of a flush write
    the same row.
    """
    if out is None:
        out = np.array(kpool, dtype=np.float64, copy=True)
    for src, dst, lo, hi, delta in runs:
        rows = kpool[:, src, :, lo:hi, :]
        out[:, dst, :, lo:hi, :] = bf16.round_bf16(rope.repos(rows, np.full(rows.shape[:-1], delta), base, layout))
    return out


def compact_copy(kpool, vpool, copies, base, layout="interleaved"):
    """Apply a compaction copy list [(src_k, src_v, src_slot, dst_k, dst_v, dst_slot, delta)] to
    copies of both pools (every layer and head): the key row is rotated by its pending delta in
    float64 and rounded to bfloat16 (copied as is when delta is 0), the value row copied."""
    ko = np.array(kpool, dtype=np.float64, copy=True)
    vo = np.array(vpool, dtype=np.float64, copy=True)
    for sk, sv, ss, dk, dv, ds, delta in copies:
        row = kpool[:, sk, :, ss, :]
        if delta:
            row = bf16.round_bf16(rope.repos(row, np.full(row.shape[:-1], delta), base, layout))
        ko[:, dk, :, ds, :] = row
        vo[:, dv, :, ds, :] = vpool[:, sv, :, ss, :]
    return ko, vo


def repos_rows_f64(kpool, layer, page, head, slot, delta, base, layout="interleaved"):
    """Unrounded float64 rotation of single rows (for the fp32-output check)."""
    rows = kpool[layer, page, head, slot, :]
    return rope.repos(rows, np.asarray(delta, np.float64), base, layout)


def gather(pool, layer, runs, which):
    """Entries [kv_len, H, d] of a segment: rows lo..hi-1 of each run's page, in order."""
    parts = [pool[layer, r[which], :, r[2]:r[3], :].transpose(1, 0, 2) for r in runs]
    return np.concatenate(parts, axis=0)


def attend_segment(q_seg, kpool, vpool, layer, runs, scale, mla=False, rows=None):
    """Segment attention over paged pools.

    q_seg [q_len, Hq, d_qk]; runs [(k_page, v_page, lo, hi)].  Under MLA the key
    is the concatenation [latent | K_pe] (d_qk = d_latent + d_pe) and the value
    is the latent.  Returns (o, lse) as oracle.attention.segment_attention.
    """
    k = gather(kpool, layer, runs, 0)
    v = gather(vpool, layer, runs, 1)
    if mla:
        k = np.concatenate([v, k], axis=-1)
    return attention.segment_attention(np.asarray(q_seg, np.float64), k, v, scale, rows=rows)


def mass_segment(q_seg, kpool, vpool, layer, runs, scale):
    """Attention mass of a segment's entries over paged pools (GQA): see attention.attention_mass."""
    k = gather(kpool, layer, runs, 0)
    return attention.attention_mass(np.asarray(q_seg, np.float64), k, scale)
