// prefill.cu -- batched causal prefill of a Qwen3-ASR-style decoder (a7, a8).
//
// Defines: "transcribe.cpp, src/arch/qwen3_asr/decoder.h", header comment
// (per-head Q/K RMSNorm over head_dim after projection and before RoPE, eps
// 1e-6; NeoX rotate_half RoPE at freq_base 1e6; GQA 16 Q / 8 KV heads of 128)
// and PrefillBuildBatched (positions shared 0..T-1, K/V written to cache rows
// [0, T), one causal mask shared by the batch); "Nest whisper-tiny,
// src/lib.linnet", DecoderLayer.prefill (write_span at 0, causal mask).
//
// a7 prep (CUDA cores, memory bound): per position t the query heads become
//   q^ = f16(RoPE_t(RMSNorm(q) * w_q)) (to the workspace), the key heads
//   k^ = f16(RoPE_t(RMSNorm(k) * w_k)) (to cache row t), V is copied to cache
//   row t and also written transposed (keys contiguous, zero-padded to a
//   multiple of 128) to the workspace, so both matrix products below read
//   K-major operands.
// a8 attention (5th-generation tensor cores): one CTA per (128-query tile,
//   sequence, query head), heaviest tiles first.  Q, K and V^T tiles arrive by
//   tiled TMA with the 128-byte swizzle; S = Q K^T and O += P V are
//   tcgen05.mma kind::f16 (f16 operands, fp32 accumulators in tensor memory,
//   256 columns: S then O).  128 threads own one query row each: they read S
//   from TMEM, run the online softmax in fp32 (log2 domain), rescale O in TMEM
//   when the row maximum grows, and write P (f16) to shared memory in the
//   swizzled K-major layout the next MMA reads.  Only key tiles at or below
//   the diagonal are visited (causal), the diagonal tile is masked.
#include <math.h>

#include <mutex>

#include "common.cuh"
#include "tcgen05.cuh"

namespace asrkv {

constexpr int kPrefillHD = 128;
constexpr int kPrepT = 16;  // positions per prep CTA
constexpr float kLog2eP = 1.4426950408889634f;

// ------------------------------------------------------------------ prep --

struct PrepArgs {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  const float* wq;
  const float* wk;
  float eps;
  int B, T, Tpad, Hq, Hkv;
  uint16_t* cache;
  int64_t seq_stride;
  uint16_t* qhat;  // [B][T][Hq*128]
  uint16_t* vt;    // [B*Hkv][128][Tpad]
  double theta[kPrefillHD / 2];
};

// grid (Tpad / kPrepT, B), 256 threads.  Shared: cos/sin of the chunk's
// positions, then the chunk's V rows for the transpose.
__global__ void __launch_bounds__(256) prefill_prep_kernel(const __grid_constant__ PrepArgs a) {
  constexpr int HD = kPrefillHD, HALF = HD / 2;
  extern __shared__ __align__(16) unsigned char psm[];
  float* cs = reinterpret_cast<float*>(psm);   // [kPrepT][HALF]
  float* sn = cs + kPrepT * HALF;              // [kPrepT][HALF]
  uint16_t* vsm = reinterpret_cast<uint16_t*>(sn + kPrepT * HALF);  // [kPrepT][Hkv*HD]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.y;
  const int t0 = blockIdx.x * kPrepT;
  const int kw = a.Hkv * HD;
  grid_launch_dependents();
  grid_dependency_wait();

  // rotation table: angle in double, reduced modulo 2*pi, then float sin/cos
  for (int idx = tid; idx < kPrepT * HALF; idx += blockDim.x) {
    const int tt = idx / HALF, i = idx % HALF;
    const double ang = (double)(t0 + tt) * a.theta[i];
    const double kq = rint(ang * 0.15915494309189535);
    double r = fma(-kq, 6.283185307179586, ang);
    r = fma(-kq, 2.4492935982947064e-16, r);
    float s, c;
    sincosf((float)r, &s, &c);
    cs[idx] = c;
    sn[idx] = s;
  }
  __syncthreads();

  // normed + roped heads: one warp per (position, head); lane l holds dims
  // 2l, 2l+1 and their RoPE partners 64+2l, 65+2l
  const int nheads = a.Hq + a.Hkv;
  for (int item = warp; item < kPrepT * nheads; item += blockDim.x >> 5) {
    const int tt = item / nheads, hh = item % nheads;
    const int t = t0 + tt;
    if (t >= a.T) continue;
    const bool is_q = hh < a.Hq;
    const int head = is_q ? hh : hh - a.Hq;
    const uint16_t* src = (is_q ? a.q + ((int64_t)b * a.T + t) * a.Hq * HD
                                : a.k + ((int64_t)b * a.T + t) * kw) + head * HD;
    const __half2 lo = *reinterpret_cast<const __half2*>(src + 2 * lane);
    const __half2 hi = *reinterpret_cast<const __half2*>(src + HALF + 2 * lane);
    const float2 xl = __half22float2(lo), xh = __half22float2(hi);
    float ss = xl.x * xl.x + xl.y * xl.y + xh.x * xh.x + xh.y * xh.y;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float rinv = 1.0f / sqrtf(ss / (float)HD + a.eps);
    const float* w = is_q ? a.wq : a.wk;
    const int i0 = 2 * lane;
    const float l0 = w[i0] * (xl.x * rinv), l1 = w[i0 + 1] * (xl.y * rinv);
    const float h0 = w[HALF + i0] * (xh.x * rinv), h1 = w[HALF + i0 + 1] * (xh.y * rinv);
    const float c0 = cs[tt * HALF + i0], s0 = sn[tt * HALF + i0];
    const float c1 = cs[tt * HALF + i0 + 1], s1 = sn[tt * HALF + i0 + 1];
    const __half2 ylo = __halves2half2(__float2half_rn(l0 * c0 - h0 * s0),
                                       __float2half_rn(l1 * c1 - h1 * s1));
    const __half2 yhi = __halves2half2(__float2half_rn(h0 * c0 + l0 * s0),
                                       __float2half_rn(h1 * c1 + l1 * s1));
    uint16_t* dst = is_q ? a.qhat + (((int64_t)b * a.T + t) * a.Hq + head) * HD
                         : a.cache + (int64_t)b * a.seq_stride + (int64_t)t * 2 * kw + head * HD;
    *reinterpret_cast<__half2*>(dst + i0) = ylo;
    *reinterpret_cast<__half2*>(dst + HALF + i0) = yhi;
  }

  // V rows: copied to the cache and staged for the transpose
  const int vec_per_row = kw / 8;
  for (int idx = tid; idx < kPrepT * vec_per_row; idx += blockDim.x) {
    const int tt = idx / vec_per_row, c = idx % vec_per_row;
    const int t = t0 + tt;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (t < a.T) {
      val = *reinterpret_cast<const uint4*>(a.v + ((int64_t)b * a.T + t) * kw + c * 8);
      *reinterpret_cast<uint4*>(a.cache + (int64_t)b * a.seq_stride + (int64_t)t * 2 * kw + kw +
                                c * 8) = val;
    }
    *reinterpret_cast<uint4*>(vsm + tt * kw + c * 8) = val;
  }
  __syncthreads();
  // V^T[b, kvh, d, t0 .. t0+16): 32 bytes per (kvh, d); zero past T
  for (int idx = tid; idx < kw; idx += blockDim.x) {
    alignas(16) uint16_t col[kPrepT];
#pragma unroll
    for (int tt = 0; tt < kPrepT; ++tt) col[tt] = vsm[tt * kw + idx];
    const int kvh = idx / HD, d = idx % HD;
    uint16_t* dst = a.vt + (((int64_t)b * a.Hkv + kvh) * HD + d) * a.Tpad + t0;
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(col);
    *reinterpret_cast<uint4*>(dst + 8) = *reinterpret_cast<const uint4*>(col + 8);
  }
}

// ------------------------------------------------------------- attention --

struct PrefillAttnArgs {
  int B, T, Hq, Hkv, n_qt;
  float sl2e;   // scale * log2(e)
  float* out;   // [B][T][Hq*128] fp32
  int32_t* dev_err;
};

constexpr int kTileBytes = 128 * 128 * 2;  // one 128 x 128 f16 operand tile
constexpr int kAttnSmem = 6 * kTileBytes + 1024 + 1024;

__global__ void __launch_bounds__(128, 1)
    prefill_attn_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                        const __grid_constant__ CUtensorMap tv, const PrefillAttnArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1024-byte alignment for the swizzled tiles
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  unsigned char* sQ = smem;                    // [2 K-halves][128 rows][128 B]
  unsigned char* sK = smem + kTileBytes;       // 2 stages
  unsigned char* sV = smem + 3 * kTileBytes;   // 2 stages (V^T: rows = dims, K = keys)
  unsigned char* sP = smem + 5 * kTileBytes;   // P: rows = queries, K = keys
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 6 * kTileBytes);  // q, kv0, kv1, mma
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 4);
  int* abort_flag = reinterpret_cast<int*>(tslot + 1);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int BH = a.B * a.Hq;
  const int qt = a.n_qt - 1 - (int)(blockIdx.x / BH);  // longest rows of tiles first
  const int rem = (int)(blockIdx.x % BH);
  const int b = rem / a.Hq, h = rem % a.Hq;
  const int kvh = h / (a.Hq / a.Hkv);
  const int q0 = qt * 128;
  const int n_kv = qt + 1;  // causal: key tiles 0 .. qt
  const int qidx = q0 + tid;  // this thread's query row

  if (tid == 0) {
    for (int i = 0; i < 4; ++i) mbar_init(&bars[i], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tslot, 256);
    tmem_relinquish();
  }
  grid_launch_dependents();
  grid_dependency_wait();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = *tslot;
  const uint32_t tS = tbase, tO = tbase + 128;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  constexpr uint32_t kIdesc = mma_idesc_f16_f32(128, 128);
  const uint32_t aQ = smem_addr(sQ), aK = smem_addr(sK), aV = smem_addr(sV), aP = smem_addr(sP);

  auto load_kv = [&](int j, int s) {
    mbar_arrive_expect_tx(&bars[1 + s], 2 * kTileBytes);
    tma_load_3d(sK + s * kTileBytes, &tk, kvh * 128, j * 128, b, &bars[1 + s]);
    tma_load_3d(sK + s * kTileBytes + kTileBytes / 2, &tk, kvh * 128 + 64, j * 128, b, &bars[1 + s]);
    tma_load_3d(sV + s * kTileBytes, &tv, j * 128, 0, b * a.Hkv + kvh, &bars[1 + s]);
    tma_load_3d(sV + s * kTileBytes + kTileBytes / 2, &tv, j * 128 + 64, 0, b * a.Hkv + kvh,
                &bars[1 + s]);
  };
  if (tid == 0) {
    mbar_arrive_expect_tx(&bars[0], kTileBytes);
    tma_load_3d(sQ, &tq, h * 128, q0, b, &bars[0]);
    tma_load_3d(sQ + kTileBytes / 2, &tq, h * 128 + 64, q0, b, &bars[0]);
    load_kv(0, 0);
    if (n_kv > 1) load_kv(1, 1);
  }

  float m_i = -INFINITY, l_i = 0.f;
  uint32_t mma_phase = 0;
  float v[32];
  for (int j = 0; j < n_kv; ++j) {
    const int s = j & 1;
    // ---- S = Q K^T
    if (tid == 0) {
      bool ok = (j > 0 || mbar_wait(&bars[0], 0)) && mbar_wait(&bars[1 + s], (j >> 1) & 1);
      if (!ok) {
        set_dev_err(a.dev_err, ASR_DEVERR_TIMEOUT);
        *abort_flag = 1;
      } else {
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * (kTileBytes / 2) + (kk & 3) * 32;
          mma_f16(tS, sw128_kmajor_desc(aQ + off), sw128_kmajor_desc(aK + s * kTileBytes + off),
                  kIdesc, kk > 0);
        }
      }
      mma_commit(&bars[3]);
    }
    if (!mbar_wait(&bars[3], mma_phase)) set_dev_err(a.dev_err, ASR_DEVERR_TIMEOUT);
    mma_phase ^= 1u;
    tc_fence_after_sync();
    const int kbase = j * 128;
    // ---- row maximum of this tile (causal mask: key <= query)
    float tmax = -INFINITY;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      tmem_ld32(tS + lane_off + c * 32, v);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (kbase + c * 32 + i <= qidx) tmax = fmaxf(tmax, v[i] * a.sl2e);
    }
    const float m_new = fmaxf(m_i, tmax);
    // ---- rescale O when the maximum grew (warp-collective TMEM access)
    const bool grow = j > 0 && m_new > m_i;
    const float alpha = grow ? exp2f(m_i - m_new) : 1.0f;
    if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        tmem_ld32(tO + lane_off + c * 32, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= alpha;
        tmem_st32(tO + lane_off + c * 32, v);
      }
      tmem_wait_st();
    }
    l_i *= alpha;
    // ---- P = exp2(S - m) as f16, written K-major with the 128-byte swizzle
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      tmem_ld32(tS + lane_off + c * 32, v);
      tmem_wait_ld();
      uint32_t packed[16];
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const float p0 = (kbase + c * 32 + i <= qidx) ? exp2f(v[i] * a.sl2e - m_new) : 0.f;
        const float p1 = (kbase + c * 32 + i + 1 <= qidx) ? exp2f(v[i + 1] * a.sl2e - m_new) : 0.f;
        l_i += p0 + p1;
        const __half2 hp = __halves2half2(__float2half_rn(p0), __float2half_rn(p1));
        packed[i / 2] = *reinterpret_cast<const uint32_t*>(&hp);
      }
      // keys c*32 .. c*32+31: K-half c/2, 16-byte chunks 4*(c%2) .. 4*(c%2)+3 of the row
      unsigned char* rowp = sP + (c >> 1) * (kTileBytes / 2) + tid * 128;
#pragma unroll
      for (int qd = 0; qd < 4; ++qd) {
        const int chunk = ((c & 1) * 4 + qd) ^ (tid & 7);
        *reinterpret_cast<uint4*>(rowp + chunk * 16) =
            make_uint4(packed[4 * qd], packed[4 * qd + 1], packed[4 * qd + 2], packed[4 * qd + 3]);
      }
    }
    m_i = m_new;
    fence_async_shared();
    tc_fence_before_sync();
    __syncthreads();
    // ---- O += P V
    if (tid == 0) {
      tc_fence_after_sync();
      if (!*abort_flag) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * (kTileBytes / 2) + (kk & 3) * 32;
          mma_f16(tO, sw128_kmajor_desc(aP + off), sw128_kmajor_desc(aV + s * kTileBytes + off),
                  kIdesc, (j > 0 || kk > 0) ? 1u : 0u);
        }
      }
      mma_commit(&bars[3]);
    }
    if (!mbar_wait(&bars[3], mma_phase)) set_dev_err(a.dev_err, ASR_DEVERR_TIMEOUT);
    mma_phase ^= 1u;
    tc_fence_after_sync();
    // stage s is free again (both products that read it are done)
    if (tid == 0 && j + 2 < n_kv && !*abort_flag) load_kv(j + 2, s);
  }

  // ---- O / l to global memory (rows past T are not written)
  const float inv = 1.0f / l_i;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    tmem_ld32(tO + lane_off + c * 32, v);
    tmem_wait_ld();
    if (qidx < a.T) {
      float* dst = a.out + (((int64_t)b * a.T + qidx) * a.Hq + h) * kPrefillHD + c * 32;
#pragma unroll
      for (int i = 0; i < 32; i += 4)
        *reinterpret_cast<float4*>(dst + i) =
            make_float4(v[i] * inv, v[i + 1] * inv, v[i + 2] * inv, v[i + 3] * inv);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tbase, 256);
  }
}

// ------------------------------------------------------------------ host --

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool make_tmap_f16_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                      uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0,
                      uint32_t box1) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  const cuuint32_t box[3] = {box0, box1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int round_up(int x, int m) { return (x + m - 1) / m * m; }

size_t prefill_ws_bytes(int B, int T, int Hq, int Hkv) {
  const size_t qhat = align_up((size_t)B * T * Hq * kPrefillHD * 2, 1024);
  const size_t vt = (size_t)B * Hkv * kPrefillHD * round_up(T, 128) * 2;
  return qhat + vt;
}

static std::once_flag g_prefill_attr;

}  // namespace asrkv

using namespace asrkv;

extern "C" int asr_prefill_attn(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                const float* q_norm_w, const float* k_norm_w, float eps,
                                float rope_base, int B, int T, int q_heads, int kv_heads,
                                int head_dim, float scale, uint16_t* cache, int64_t seq_stride,
                                int capacity, float* out, void* ws, size_t ws_bytes,
                                int32_t* dev_err, asr_stream_t stream) {
  if (B < 0 || B > ASR_MAX_BATCH || T < 1 || q_heads < 1 || kv_heads < 1 || capacity < 1 ||
      !(eps >= 0.f) || !(rope_base > 0.f))
    return ASR_ERR_INVALID_ARG;
  if (head_dim != kPrefillHD || q_heads % kv_heads != 0 || kv_heads > 16 || q_heads > 64)
    return ASR_ERR_UNSUPPORTED;
  if (T > capacity) return ASR_ERR_INVALID_ARG;
  if (B == 0) return ASR_OK;
  if (!q || !k || !v || !q_norm_w || !k_norm_w || !cache || !out) return ASR_ERR_INVALID_ARG;
  const int64_t row = 2LL * kv_heads * head_dim;
  if (seq_stride < (int64_t)capacity * row) return ASR_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(cache) || !aligned16(out) ||
      seq_stride % 8 != 0)
    return ASR_ERR_MISALIGNED;
  if ((int64_t)B * T * q_heads * head_dim >= (1LL << 40)) return ASR_ERR_UNSUPPORTED;
  if (!ws || ((uintptr_t)ws & 255u) != 0 || ws_bytes < prefill_ws_bytes(B, T, q_heads, kv_heads))
    return ASR_ERR_WORKSPACE;
  const int Tpad = round_up(T, 128);
  uint16_t* qhat = static_cast<uint16_t*>(ws);
  uint16_t* vt = reinterpret_cast<uint16_t*>(static_cast<char*>(ws) +
                                             align_up((size_t)B * T * q_heads * kPrefillHD * 2, 1024));
  cudaError_t attr = cudaSuccess;
  std::call_once(g_prefill_attr, [&] {
    attr = cudaFuncSetAttribute(prefill_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kAttnSmem);
    if (attr == cudaSuccess)
      attr = cudaFuncSetAttribute(prefill_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  100 * 1024);
  });
  if (attr != cudaSuccess) return ASR_ERR_CUDA;

  // tensor maps: q^ (dims: Hq*128, T, B), cache (row, capacity, B), V^T (Tpad, 128, B*Hkv)
  CUtensorMap tq, tk, tv;
  if (!make_tmap_f16_3d(&tq, qhat, (uint64_t)q_heads * kPrefillHD, T, B,
                        (uint64_t)q_heads * kPrefillHD * 2, (uint64_t)T * q_heads * kPrefillHD * 2,
                        64, 128) ||
      !make_tmap_f16_3d(&tk, cache, (uint64_t)row, capacity, B, (uint64_t)row * 2,
                        (uint64_t)seq_stride * 2, 64, 128) ||
      !make_tmap_f16_3d(&tv, vt, Tpad, kPrefillHD, (uint64_t)B * kv_heads, (uint64_t)Tpad * 2,
                        (uint64_t)Tpad * kPrefillHD * 2, 64, 128))
    return ASR_ERR_CUDA;

  PrepArgs pa = {};
  pa.q = q;
  pa.k = k;
  pa.v = v;
  pa.wq = q_norm_w;
  pa.wk = k_norm_w;
  pa.eps = eps;
  pa.B = B;
  pa.T = T;
  pa.Tpad = Tpad;
  pa.Hq = q_heads;
  pa.Hkv = kv_heads;
  pa.cache = cache;
  pa.seq_stride = seq_stride;
  pa.qhat = qhat;
  pa.vt = vt;
  for (int i = 0; i < kPrefillHD / 2; ++i)
    pa.theta[i] = pow((double)rope_base, -2.0 * i / kPrefillHD);
  const size_t prep_smem =
      2 * kPrepT * (kPrefillHD / 2) * sizeof(float) + (size_t)kPrepT * kv_heads * kPrefillHD * 2;
  cudaError_t e = launch_pdl(prefill_prep_kernel, dim3(Tpad / kPrepT, B), dim3(256), prep_smem,
                             (cudaStream_t)stream, pa);
  if (e != cudaSuccess) return ASR_ERR_CUDA;

  PrefillAttnArgs aa = {};
  aa.B = B;
  aa.T = T;
  aa.Hq = q_heads;
  aa.Hkv = kv_heads;
  aa.n_qt = (T + 127) / 128;
  aa.sl2e = scale * kLog2eP;
  aa.out = out;
  aa.dev_err = dev_err;
  e = launch_pdl(prefill_attn_kernel, dim3(aa.n_qt * B * q_heads), dim3(128), (size_t)kAttnSmem,
                 (cudaStream_t)stream, tq, tk, tv, aa);
  return e == cudaSuccess ? ASR_OK : ASR_ERR_CUDA;
}
