// kv_write: scatter the K and V rows of newly appended (or stub) tokens into
// their pool pages.  [AKV-notes] section 1 "Problem & Solution": append adds
// the KV state of new tokens; the paged layout is the engine's.
//
//   src  bf16 [L][n][H][D]              (the model's per-layer output order)
//   pool bf16 [L][P][H][page][D]
//   rows int32[n] = page * page_size + slot of each token
//
// One launch moves both tensors (blockIdx.y: 0 = K, 1 = V).  One thread moves
// one 16-byte vector; consecutive threads read consecutive source bytes, so
// the loads are fully coalesced and each D-row lands as D/8 contiguous vectors
// of one pool row.  HBM-bound: 2 x (L n H (D_k + D_v) x 2 B); for a turn's
// few MiB the launch ramp dominates, so index arithmetic stays in 32 bits
// whenever the element count allows.
#include <cuda_bf16.h>

#include "akv_internal.h"

namespace akv {
namespace {

struct KvSide {
  const uint4* src;
  uint4* pool;
  const int32_t* rows;
  int vec_per_row;
};

template <typename I>
__global__ void __launch_bounds__(256) kv_write_kernel(KvSide k, KvSide v, I n, int n_layers, int heads, int page,
                                                       int64_t n_pages, DevErr* err) {
  const KvSide s = blockIdx.y == 0 ? k : v;
  const I vpr = I(s.vec_per_row);
  const I total = I(n_layers) * n * I(heads) * vpr;
  const int64_t row_vecs = int64_t(page) * s.vec_per_row;  // one (page, head) block
  const int64_t page_vecs = row_vecs * heads;              // one page, all heads
  const int64_t layer_vecs = page_vecs * n_pages;
  for (I i = I(blockIdx.x) * I(blockDim.x) + I(threadIdx.x); i < total; i += I(gridDim.x) * I(blockDim.x)) {
    const I vv = i % vpr;
    I rest = i / vpr;
    const I h = rest % I(heads);
    rest /= I(heads);
    const I t = rest % n;
    const I l = rest / n;
    const int32_t r = __ldg(s.rows + t);
#ifdef AKV_CHECKED
    if (r < 0 || int64_t(r) >= n_pages * page) {  // skip the row: it names no slot of the pool
      report_device_error(err, 2, int(t), r);
      continue;
    }
#endif
    const int32_t pg = r / page, slot = r % page;
    const uint4 x = __ldcs(s.src + i);
    __stcs(s.pool + int64_t(l) * layer_vecs + int64_t(pg) * page_vecs + int64_t(h) * row_vecs +
               int64_t(slot) * s.vec_per_row + int64_t(vv),
           x);
  }
}

}  // namespace

cudaError_t launch_kv_write(const void* src_k, void* pool_k, const int32_t* rows_k, int dim_k, const void* src_v,
                            void* pool_v, const int32_t* rows_v, int dim_v, int64_t n, int n_layers, int heads,
                            int page, int64_t n_pages, int n_sm, DevErr* err, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  if (dim_k % 8 || dim_v % 8) return cudaErrorInvalidValue;
  const int64_t total = int64_t(n_layers) * n * heads * (std::max(dim_k, dim_v) / 8);
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, int64_t(n_sm) * 8);
  const KvSide k{static_cast<const uint4*>(src_k), static_cast<uint4*>(pool_k), rows_k, dim_k / 8};
  const KvSide v{static_cast<const uint4*>(src_v), static_cast<uint4*>(pool_v), rows_v, dim_v / 8};
  const dim3 grid(unsigned(blocks), 2);
  if (total < (int64_t(1) << 31) - int64_t(blocks) * 256)
    kv_write_kernel<int32_t><<<grid, 256, 0, st>>>(k, v, int32_t(n), n_layers, heads, page, n_pages, err);
  else
    kv_write_kernel<int64_t><<<grid, 256, 0, st>>>(k, v, n, n_layers, heads, page, n_pages, err);
  return cudaGetLastError();
}

}  // namespace akv
