// kv_ops.cu -- K/V append (a1) and beam reorder (a6).
//
// Both are pure data movement: the append converts one fp32 row per sequence
// to f16 (round to nearest even) and scatters it into its cache slot; the
// reorder gathers whole history blocks of beams into a second cache buffer.
// Each thread moves 16-byte vectors; rows of one (sequence, layer) are
// contiguous, so every warp touches contiguous 512-byte spans.
#include "common.cuh"

namespace asrkv {

// ------------------------------------------------------------- append ----
// "wavo 0.1.0, src/whisper/decoder.rs", Decoder::record_step: k and v of the
// new token become f16 row `pos` of the layer's cache.
__global__ void __launch_bounds__(256) kv_append_kernel(
    const float* __restrict__ k, const float* __restrict__ v, int64_t src_row_stride,
    uint16_t* __restrict__ cache, int64_t seq_stride, const int32_t* __restrict__ slot, int B,
    int half_elems, int capacity, int32_t* dev_err) {
  grid_launch_dependents();  // the next kernel may launch; it waits for our completion
  grid_dependency_wait();
  const int vec_per_half = half_elems >> 3;  // 8 f16 per 16-byte vector
  const int64_t total = (int64_t)B * 2 * vec_per_half;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int b = (int)(i / (2 * vec_per_half));
    const int w = (int)(i % (2 * vec_per_half));  // vector within the row
    const int s = slot[b];
    if (s < 0 || s >= capacity) {
      if (w == 0) set_dev_err(dev_err, ASR_DEVERR_LEN);
      continue;
    }
    const bool is_v = w >= vec_per_half;
    const int e = (is_v ? w - vec_per_half : w) * 8;
    const float* src = (is_v ? v : k) + (int64_t)b * src_row_stride + e;
    float f[8];
    const float4 a = *reinterpret_cast<const float4*>(src);
    const float4 c = *reinterpret_cast<const float4*>(src + 4);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = c.x; f[5] = c.y; f[6] = c.z; f[7] = c.w;
    uint16_t* dst = cache + (int64_t)b * seq_stride + (int64_t)s * 2 * half_elems +
                    (is_v ? half_elems : 0) + e;
    *reinterpret_cast<uint4*>(dst) = f8_to_h8(f);
  }
  grid_launch_dependents();
}

// ---------------------------------------------------------- rearrange ----
// "mlx-bun whisper.ts", WhisperKvCache.rearrange: every layer's self k/v keep
// the rows of beam idx[b] (take along the batch axis).
//
// Grid: x strides over the 16-byte vectors of one (beam, layer) block; y is
// beam * n_layers + layer.  Each thread keeps kUnroll loads in flight.
constexpr int kRearrangeThreads = 256;
constexpr int kRearrangeUnroll = 4;

__global__ void __launch_bounds__(kRearrangeThreads) kv_rearrange_kernel(
    const uint16_t* __restrict__ src, uint16_t* __restrict__ dst, int64_t seq_stride,
    int64_t layer_stride, int n_layers, int row_elems, int capacity,
    const int32_t* __restrict__ idx, const int32_t* __restrict__ lens_src,
    int32_t* __restrict__ lens_dst, int B, int32_t* dev_err) {
  grid_launch_dependents();  // the next kernel may launch; it waits for our completion
  grid_dependency_wait();
  const int b = blockIdx.y / n_layers;
  const int l = blockIdx.y % n_layers;
  const int s = idx[b];
  const bool idx_ok = s >= 0 && s < B;
  const int len = idx_ok ? lens_src[s] : 0;
  const bool ok = idx_ok && len >= 1 && len <= capacity;
  if (blockIdx.x == 0 && l == 0 && threadIdx.x == 0) {
    lens_dst[b] = ok ? len : 0;
    if (!ok) set_dev_err(dev_err, idx_ok ? ASR_DEVERR_LEN : ASR_DEVERR_INDEX);
  }
  if (!ok) {
    grid_launch_dependents();
    return;
  }
  const int64_t nvec = (int64_t)(len - 1) * row_elems / 8;
  const uint4* from = reinterpret_cast<const uint4*>(src + (int64_t)s * seq_stride +
                                                     (int64_t)l * layer_stride);
  uint4* to = reinterpret_cast<uint4*>(dst + (int64_t)b * seq_stride + (int64_t)l * layer_stride);
  const int64_t step = (int64_t)gridDim.x * kRearrangeThreads;
  for (int64_t base = (int64_t)blockIdx.x * kRearrangeThreads + threadIdx.x; base < nvec;
       base += step * kRearrangeUnroll) {
    uint4 t[kRearrangeUnroll];
#pragma unroll
    for (int u = 0; u < kRearrangeUnroll; ++u) {
      const int64_t i = base + u * step;
      if (i < nvec) t[u] = __ldcs(from + i);
    }
#pragma unroll
    for (int u = 0; u < kRearrangeUnroll; ++u) {
      const int64_t i = base + u * step;
      if (i < nvec) to[i] = t[u];
    }
  }
  grid_launch_dependents();
}

}  // namespace asrkv

using namespace asrkv;

extern "C" int asr_kv_append(const float* k, const float* v, int64_t src_row_stride,
                             uint16_t* cache, int64_t seq_stride, const int32_t* slot, int B,
                             int kv_heads, int head_dim, int capacity, int32_t* dev_err,
                             asr_stream_t stream) {
  if (B < 0 || B > ASR_MAX_BATCH || kv_heads < 1 || capacity < 1 || head_dim < 1)
    return ASR_ERR_INVALID_ARG;
  if (head_dim % 8 != 0 || kv_heads > ASR_MAX_KV_HEADS) return ASR_ERR_UNSUPPORTED;
  if (B == 0) return ASR_OK;
  if (!k || !v || !cache || !slot) return ASR_ERR_INVALID_ARG;
  const int64_t half = (int64_t)kv_heads * head_dim;
  if (src_row_stride < half || seq_stride < (int64_t)capacity * 2 * half)
    return ASR_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(cache) || src_row_stride % 4 != 0 ||
      seq_stride % 8 != 0)
    return ASR_ERR_MISALIGNED;
  const int64_t total = (int64_t)B * 2 * (half / 8);
  const int threads = 256;
  const int blocks = (int)ceil_div64(total, threads);
  cudaError_t e = launch_pdl(kv_append_kernel, dim3(blocks), dim3(threads), 0,
                             (cudaStream_t)stream, k, v, src_row_stride, cache, seq_stride, slot, B,
                             (int)half, capacity, dev_err);
  return e == cudaSuccess ? ASR_OK : ASR_ERR_CUDA;
}

extern "C" int asr_kv_rearrange(const uint16_t* src, uint16_t* dst, int64_t seq_stride,
                                int64_t layer_stride, int n_layers, int row_elems, int capacity,
                                const int32_t* idx, const int32_t* lens_src, int32_t* lens_dst,
                                int B, int32_t* dev_err, asr_stream_t stream) {
  if (B < 0 || B > ASR_MAX_BATCH || n_layers < 1 || row_elems < 8 || capacity < 1)
    return ASR_ERR_INVALID_ARG;
  if (B == 0) return ASR_OK;
  if (!src || !dst || !idx || !lens_src || !lens_dst) return ASR_ERR_INVALID_ARG;
  if (layer_stride < (int64_t)capacity * row_elems ||
      seq_stride < (int64_t)(n_layers - 1) * layer_stride + (int64_t)capacity * row_elems)
    return ASR_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(dst) || row_elems % 8 != 0 || seq_stride % 8 != 0 ||
      layer_stride % 8 != 0)
    return ASR_ERR_MISALIGNED;
  const uintptr_t bytes = (uintptr_t)B * (uintptr_t)seq_stride * 2;
  const uintptr_t s0 = (uintptr_t)src, d0 = (uintptr_t)dst;
  if (s0 < d0 + bytes && d0 < s0 + bytes) return ASR_ERR_ALIAS;
  if ((int64_t)B * n_layers > 65535) return ASR_ERR_UNSUPPORTED;
  // x covers one (beam, layer) block of at most capacity rows
  const int64_t max_vec = (int64_t)capacity * row_elems / 8;
  int gx = (int)ceil_div64(max_vec, (int64_t)kRearrangeThreads * kRearrangeUnroll);
  if (gx < 1) gx = 1;
  dim3 grid(gx, B * n_layers);
  cudaError_t e = launch_pdl(kv_rearrange_kernel, grid, dim3(kRearrangeThreads), 0,
                             (cudaStream_t)stream, src, dst, seq_stride, layer_stride, n_layers,
                             row_elems, capacity, idx, lens_src, lens_dst, B, dev_err);
  return e == cudaSuccess ? ASR_OK : ASR_ERR_CUDA;
}
