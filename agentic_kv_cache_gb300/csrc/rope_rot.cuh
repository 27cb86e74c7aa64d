// The rotation arithmetic of a repositioned key, shared by every kernel that
// rotates stored keys (repos_rotate materialises it in the pool; the fused
// attention path applies it to a K tile in shared memory), so both give the
// same bf16 bits: x' = R(delta * theta_j) x per pair in float32 with the
// (cos, sin) of a host-built float64 table rounded to float32, then one
// round-to-nearest-even to bf16.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

namespace akv {

__device__ __forceinline__ float2 rot2(uint32_t xy, float c, float s) {
  __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&xy);
  const float2 f = __bfloat1622float2(b);
  return make_float2(fmaf(c, f.x, -s * f.y), fmaf(s, f.x, c * f.y));
}

__device__ __forceinline__ uint32_t pack_rot(float2 y) {
  __nv_bfloat162 r = __floats2bfloat162_rn(y.x, y.y);
  return *reinterpret_cast<uint32_t*>(&r);
}

// Both halves of a (j, j + D/2) pair: a holds first-half elements e, e+1; b
// the matching second-half elements.
__device__ __forceinline__ void rot_halves(uint32_t a, uint32_t b, float c0, float s0, float c1, float s1,
                                           float2& ya, float2& yb) {
  __nv_bfloat162 ab = *reinterpret_cast<__nv_bfloat162*>(&a);
  __nv_bfloat162 bb = *reinterpret_cast<__nv_bfloat162*>(&b);
  const float2 fa = __bfloat1622float2(ab), fb = __bfloat1622float2(bb);
  ya = make_float2(fmaf(c0, fa.x, -s0 * fb.x), fmaf(c1, fa.y, -s1 * fb.y));
  yb = make_float2(fmaf(s0, fa.x, c0 * fb.x), fmaf(s1, fa.y, c1 * fb.y));
}

}  // namespace akv
