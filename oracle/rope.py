"""RoPE and the repos primitive in float64 (test infrastructure only).

[AKV-blog] section 2, "The Repos Primitive and Rotary Position Embeddings":
RoPE rotates each 2-D component of a key or query at position m by
R(m*theta) = [[cos, -sin], [sin, cos]].  Because these rotations form SO(2),
R(a) R(b) = R(a+b), so a key cached at position m is moved to another
position by one extra rotation of the stored vector, with no access to the
hidden states.  [Leyline] "Method" writes the same thing with a signed shift:
every downstream slot moves by Delta and its K_pe becomes R(Delta) * K_pe.

Conventions fixed here (the pages leave them open):

* Delta is signed, new_position = old_position + Delta ([Leyline] "Method").
  The blog's R_{-Delta} for a drop of length Delta is this with Delta -> -Delta.
* theta_j = base ** (-2 j / d_rot) for j in [0, d_rot/2); the pages never
  define Theta beyond "theta", so no frequency scaling is applied.
* Pairing: "interleaved" pairs (2j, 2j+1), as the blog's 2x2 formula and its
  kernel listing in section 5 do.  "half" pairs (j, j + d_rot/2) is the other
  common layout, kept behind a flag.
"""
import numpy as np


def theta(d_rot, base):
    """Per-pair RoPE frequencies theta_j = base**(-2j/d_rot), float64, shape [d_rot/2]."""
    if d_rot % 2:
        raise ValueError("rotated dimension must be even")
    j = np.arange(d_rot // 2, dtype=np.float64)
    return np.power(float(base), -2.0 * j / d_rot)


def pair_indices(d_rot, layout):
    """Index arrays (first, second) of the 2-D components that rotate together."""
    j = np.arange(d_rot // 2)
    if layout == "interleaved":
        return 2 * j, 2 * j + 1
    if layout == "half":
        return j, j + d_rot // 2
    raise ValueError(f"unknown RoPE layout {layout!r}")


def rotate(x, angle, layout="interleaved"):
    """Apply R(angle_j) = [[cos, -sin], [sin, cos]] to every pair j of x.

    x: [..., d_rot] float64; angle: [..., d_rot/2] (broadcast against x).
    """
    x = np.asarray(x, dtype=np.float64)
    a, b = pair_indices(x.shape[-1], layout)
    c, s = np.cos(angle), np.sin(angle)
    out = np.empty(np.broadcast_shapes(x.shape, np.shape(angle)[:-1] + x.shape[-1:]))
    xa, xb = x[..., a], x[..., b]
    out[..., a] = c * xa - s * xb
    out[..., b] = s * xa + c * xb
    return out


def rope(x, pos, base, layout="interleaved"):
    """RoPE of vectors x (last axis d_rot) at integer positions pos (shape x.shape[:-1])."""
    x = np.asarray(x, dtype=np.float64)
    pos = np.asarray(pos, dtype=np.float64)
    th = theta(x.shape[-1], base)
    return rotate(x, pos[..., None] * th, layout)


def repos(k, delta, base, layout="interleaved"):
    """The repos primitive: move keys already rotated at p to p + delta, k' = R(delta*theta) k."""
    k = np.asarray(k, dtype=np.float64)
    delta = np.asarray(delta, dtype=np.float64)
    th = theta(k.shape[-1], base)
    return rotate(k, delta[..., None] * th, layout)
