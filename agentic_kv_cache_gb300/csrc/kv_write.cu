// kv_write: scatter the K or V rows of newly appended (or stub) tokens into
// their pool pages.  [AKV-notes] section 1 "Problem & Solution": append adds
// the KV state of new tokens; the paged layout is the engine's.
//
//   src  bf16 [L][n][H][D]              (the model's per-layer output order)
//   pool bf16 [L][P][H][page][D]
//   rows int32[n] = page * page_size + slot of each token
//
// One thread moves one 16-byte vector; consecutive threads read consecutive
// source bytes, so the loads are fully coalesced and each D-row lands as
// D/8 contiguous vectors of one pool row.  HBM-bound: 2 x (L n H D x 2 B).
#include <cuda_bf16.h>

#include "akv_internal.h"

namespace akv {
namespace {

__global__ void __launch_bounds__(256) kv_write_kernel(const uint4* __restrict__ src, uint4* __restrict__ pool,
                                                       const int32_t* __restrict__ rows, int64_t n, int n_layers,
                                                       int heads, int vec_per_row, int page, int64_t n_pages) {
  const int64_t total = int64_t(n_layers) * n * heads * vec_per_row;
  const int64_t row_vecs = int64_t(page) * vec_per_row;         // one (page, head) block
  const int64_t page_vecs = row_vecs * heads;                   // one page, all heads
  const int64_t layer_vecs = page_vecs * n_pages;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
    const int v = int(i % vec_per_row);
    int64_t rest = i / vec_per_row;
    const int h = int(rest % heads);
    rest /= heads;
    const int64_t t = rest % n;
    const int64_t l = rest / n;
    const int32_t r = __ldg(rows + t);
    const int64_t pg = r / page, slot = r % page;
    const uint4 x = __ldcs(src + i);
    __stcs(pool + l * layer_vecs + pg * page_vecs + h * row_vecs + slot * vec_per_row + v, x);
  }
}

}  // namespace

cudaError_t launch_kv_write(const void* src, void* pool, const int32_t* rows, int64_t n, int n_layers, int heads,
                            int dim, int page, int64_t n_pages, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  if (dim % 8) return cudaErrorInvalidValue;
  const int64_t total = int64_t(n_layers) * n * heads * (dim / 8);
  int sms = 152;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, int64_t(sms) * 16);
  kv_write_kernel<<<unsigned(blocks), 256, 0, st>>>(static_cast<const uint4*>(src), static_cast<uint4*>(pool), rows,
                                                    n, n_layers, heads, dim / 8, page, n_pages);
  return cudaGetLastError();
}

}  // namespace akv
