// linear.cu -- the dense steps of a decoder layer around the attention (next
// row): LayerNorm, then the product of the activations with an f16 weight,
// with a Bias, Residual or Gelu epilogue.
//
// Defines: "wavo 0.1.0, src/whisper/decoder.rs", Decoder::record_step
// (layer_norm of x into y; gemv of y with the qkv, self_out, cross_q,
// cross_out, fc1 and fc2 weights, epilogue Bias, Residual(1.0) or Gelu);
// "Nest whisper-tiny, src/lib.linnet", LayerNorm (eps 1e-5) and Mlp (fc2 of
// gelu_erf of fc1).
//
//   a_m  = LayerNorm(x_m) * g + b      (or x_m when no LayerNorm is asked)
//   v_mn = sum_k a_mk W[n][k] + bias_n
//   y_mn = v_mn | y_mn + v_mn | v_mn * Phi(v_mn)
//
// For one token per sequence this is weight-bound: M (the sequences) is tens
// of rows while W is megabytes, read once.  The kernel streams W through a
// TMA ring and puts the product on the tensor cores with the operands
// swapped: D[n][m] = W[n][:] . a[m][:], so the 128 rows of one MMA are 128
// weight rows and the batch is the MMA's N (16..256), with no padded rows.
// The activations keep their fp32 precision: each is split into an f16 high
// part and an f16 remainder, a = hi + lo, and both are multiplied by the f16
// weight into the same fp32 accumulator (two MMAs per K step; the tensor
// core is idle most of the time here anyway).
//
// Work split: 128 weight rows x a range of K per CTA.  With few weight rows
// (N = 1280 is ten tiles) the K axis is split until the grid covers the GPU;
// the CTAs of one tile add their partial sums into a zero fp32 tile in the
// workspace (red.add), and the last to arrive (a counter per tile) applies
// the epilogue, writes y and puts the tile and the counter back to zero.
//
// LayerNorm without a pass over whole rows: a CTA only sees its K range, so
// the normalisation is folded into the product.  With x_0 the row's first
// element, the operand is (x_k - x_0) * g_k, and two more operand rows hold g
// and b, so the same accumulator collects cn = sum_k g_k W_nk and dn =
// sum_k b_k W_nk; the CTA also sums (x_k - x_0) and its square over its K
// range.  Once all K is in (after the split reduction), mean - x_0 = s1/K,
// var = s2/K - (s1/K)^2 and
//   sum_k a_mk W_nk = rstd * (sum_k (x_k - x_0) g_k W_nk - (mean - x_0) cn) + dn.
// Shifting by x_0 keeps both differences of the size of the row's spread.
//
// Roles: warp 4 streams W (128 rows x 64 k per stage, 128-byte swizzle) and
// holds the TMEM allocation; warp 5 issues tcgen05.mma; warps 0-3 write the
// hi/lo operand to shared memory in the same swizzled layout (with the
// LayerNorm sums), then drain the accumulator (thread = weight row, one TMEM
// lane each) and run the epilogue.  W is never written by a kernel of this
// library, so the weight loads start before the wait on the previous grid
// (programmatic dependent launch): they overlap its tail.
#include <mutex>

#include "common.cuh"
#include "tcgen05.cuh"

namespace asrkv {

constexpr int kLinStages = 4;
constexpr int kLinWTile = 128 * 64 * 2;  // 16 KB: 128 weight rows x 64 k
constexpr int kLinThreads = 192;         // warps 0-3 operand + epilogue, 4 TMA, 5 MMA
constexpr int kLinMaxMT = 256;           // the MMA's N
constexpr int kLinXCap = 96 * 1024;      // both activation planes of one CTA
constexpr int kLinSmemFixed = 1024 + kLinStages * kLinWTile + 256 + 4 * kLinMaxMT * 4;

struct LinArgs {
  const float* x;
  int64_t x_stride;
  const float* ln_g;
  const float* ln_b;
  float eps;
  const float* bias;
  float* y;
  int64_t y_stride;
  float* acc;         // [tiles][MT][128] fp32, zero between calls
  float* stats;       // [tiles][MT][2] fp32 (LayerNorm sums), zero between calls
  uint32_t* tickets;  // [tiles], zero between calls
  int M, N, K, mode;
  int MT, MR, n_tiles, S, KB, nkb_max;  // MR: sequences per tile (MT - 2 or fewer with LayerNorm)
  uint32_t tmem_cols;
  int32_t* dev_err;
};

__device__ __forceinline__ float lin_epilogue(int mode, float v, float yold) {
  if (mode == ASR_LINEAR_RESIDUAL) return yold + v;
  if (mode == ASR_LINEAR_GELU) return 0.5f * v * (1.0f + erff(v * 0.70710678118654752f));
  return v;
}

// Row statistics of the LayerNorm from the K-sums of the values shifted by
// the row's first element x_0: s1 = sum (x - x_0), s2 = sum (x - x_0)^2.
// dm = mean - x_0 and rstd = 1 / sqrt(var + eps), var = s2/K - (s1/K)^2.
__device__ __forceinline__ void lin_row_stats(float s1, float s2, float inv_k, float eps, int t,
                                              float* s_dm, float* s_rs) {
  const float dm = s1 * inv_k;
  const float var = fmaxf(s2 * inv_k - dm * dm, 0.f);
  s_dm[t] = dm;
  s_rs[t] = rsqrtf(var + eps);
}

// Outputs (m_first + e, n) for e < cnt from the K-sums v[e]:
//   LayerNorm: a_mk = ((x_mk - x_0) - dm) * rstd * g_k + b_k, so
//   sum_k a_mk W_nk = rstd * (v - dm * cn) + dn with cn = sum_k g_k W_nk and
//   dn = sum_k b_k W_nk; otherwise the sum is v itself.  Then bias, epilogue.
// The old values of a residual are loaded before any store.
__device__ __forceinline__ void lin_emit16(const LinArgs& a, int m_first, int cnt, int n,
                                           const float* v, float bn, bool ln, const float* dm,
                                           const float* rs, float cn, float dn) {
  if (n >= a.N) return;
  float yo[16];
  if (a.mode == ASR_LINEAR_RESIDUAL) {
#pragma unroll
    for (int e = 0; e < 16; ++e)
      yo[e] = e < cnt ? a.y[(int64_t)(m_first + e) * a.y_stride + n] : 0.f;
  }
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    if (e < cnt) {
      const float t = ln ? rs[e] * (v[e] - dm[e] * cn) + dn : v[e];
      a.y[(int64_t)(m_first + e) * a.y_stride + n] = lin_epilogue(a.mode, t + bn, yo[e]);
    }
  }
}

__global__ void __launch_bounds__(kLinThreads, 1)
linear_kernel(const __grid_constant__ CUtensorMap tw, const LinArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int MT = a.MT;
  const int plane = MT * 128 * a.nkb_max;                  // bytes of one activation plane
  unsigned char* sW = smem;                                // stages x 16 KB
  unsigned char* sXh = sW + kLinStages * kLinWTile;        // hi plane: [nkb][MT rows][128 B]
  unsigned char* sXl = sXh + plane;                        // lo plane
  uint64_t* full = reinterpret_cast<uint64_t*>(sXl + plane);
  uint64_t* empty = full + kLinStages;
  uint64_t* x_full = empty + kLinStages;   // the activation operand is in shared memory
  uint64_t* acc_full = x_full + 1;         // the accumulator is complete
  uint32_t* tslot = reinterpret_cast<uint32_t*>(acc_full + 1);
  int* last_flag = reinterpret_cast<int*>(tslot + 1);
  int* abort_flag = last_flag + 1;  // a wait of warps 0-3 gave up
  float* s_s1 = reinterpret_cast<float*>(smem + kLinStages * kLinWTile + 2 * plane + 256);
  float* s_s2 = s_s1 + kLinMaxMT;  // LayerNorm sums of this CTA's K range
  float* s_dm = s_s2 + kLinMaxMT;  // mean - x_0 of each row
  float* s_rs = s_dm + kLinMaxMT;  // 1 / sqrt(var + eps)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int u = blockIdx.x;
  const int s = u % a.S, tile = u / a.S;
  const int nt = tile % a.n_tiles, mt = tile / a.n_tiles;
  const int kb0 = (int)((int64_t)s * a.KB / a.S);
  const int nkb = (int)((int64_t)(s + 1) * a.KB / a.S) - kb0;
  const int m0 = mt * a.MR, n0 = nt * 128;
  const int Mv = min(a.MR, a.M - m0);

  if (tid == 0) {
    for (int i = 0; i < kLinStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(x_full, 128);
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 4) {
    tmem_alloc(tslot, a.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = *tslot;
  grid_launch_dependents();
  bool ok = true;

  if (warp == 4) {
    // ================================================ W producer (no wait)
    int j = 0;
    for (; j < nkb; ++j) {
      const int st = j % kLinStages;
      if (j >= kLinStages && !(ok = mbar_wait_warp(&empty[st], ((j / kLinStages) - 1) & 1))) break;
      mbar_arrive_expect_tx_warp(&full[st], kLinWTile);
      tma_load_3d_warp(sW + st * kLinWTile, &tw, (kb0 + j) * 64, n0, 0, &full[st]);
    }
    // every issued copy has landed before the CTA may leave
    for (int i = max(0, j - kLinStages); i < j; ++i)
      if (!mbar_wait_warp(&full[i % kLinStages], (i / kLinStages) & 1)) ok = false;
  } else if (warp == 5) {
    // ================================================ MMA issuer
    const uint32_t idesc = mma_idesc_f16_f32(128, MT);
    const uint32_t aW = smem_addr(sW), aH = smem_addr(sXh), aL = smem_addr(sXl);
    ok = mbar_wait_warp(x_full, 0);
    tc_fence_after_sync();
    for (int j = 0; j < nkb && ok; ++j) {
      const int st = j % kLinStages;
      ok = mbar_wait_warp(&full[st], (j / kLinStages) & 1);
      tc_fence_after_sync();
      if (!ok) break;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t wd = sw128_kmajor_desc(aW + st * kLinWTile + kk * 32);
        const uint32_t xo = (uint32_t)(j * MT * 128 + kk * 32);
        mma_f16_warp(tbase, wd, sw128_kmajor_desc(aH + xo), idesc, (j > 0 || kk > 0) ? 1u : 0u);
        mma_f16_warp(tbase, wd, sw128_kmajor_desc(aL + xo), idesc, 1u);
      }
      mma_commit_warp(&empty[st]);
    }
    if (ok) mma_commit_warp(acc_full);
  } else {
    // ================================================ operand + epilogue
    grid_dependency_wait();  // x (and y, the workspace) belong to earlier grids
    const bool ln = a.ln_g != nullptr;
    if (ln) {
      for (int i = tid; i < MT; i += 128) s_s1[i] = s_s2[i] = 0.f;
      named_bar(1, 128);
    }
    // The operand: MT rows x nkb k-blocks x eight 16-byte chunks; chunk c of
    // row r sits at c ^ (r % 8) (the 128-byte swizzle the MMA reads).  Rows
    // < Mv: the activations (LayerNorm: (x - x_0) * g, see the epilogue);
    // with LayerNorm, row Mv holds g and row Mv+1 holds b, so that the
    // accumulator also collects sum_k g_k W_nk and sum_k b_k W_nk; the rest
    // is zero.  Loads of four items are issued before any is used.
    const int items = MT * nkb * 8;  // a multiple of 128: warp-uniform batches
    for (int i0 = tid; i0 < items; i0 += 4 * 128) {
      float4 xv[4][2], gv[4][2];
      float shv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = i0 + q * 128;
        const int c = i & 7, j = (i >> 3) % nkb, r = (i >> 3) / nkb;
        const int k = (kb0 + j) * 64 + c * 8;
        xv[q][0] = xv[q][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        gv[q][0] = gv[q][1] = xv[q][0];
        shv[q] = 0.f;
        if (i < items) {
          const float* src = nullptr;
          if (r < Mv) {
            src = a.x + (int64_t)(m0 + r) * a.x_stride + k;
            if (ln) {
              shv[q] = __ldg(a.x + (int64_t)(m0 + r) * a.x_stride);
              gv[q][0] = __ldg(reinterpret_cast<const float4*>(a.ln_g + k));
              gv[q][1] = __ldg(reinterpret_cast<const float4*>(a.ln_g + k + 4));
            }
          } else if (ln && r == Mv) {
            src = a.ln_g + k;
          } else if (ln && r == Mv + 1) {
            src = a.ln_b + k;
          }
          if (src) {
            xv[q][0] = __ldg(reinterpret_cast<const float4*>(src));
            xv[q][1] = __ldg(reinterpret_cast<const float4*>(src + 4));
          }
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = i0 + q * 128;
        if (i >= items) break;  // uniform across the warp
        const int c = i & 7, j = (i >> 3) % nkb, r = (i >> 3) / nkb;
        float f[8] = {xv[q][0].x, xv[q][0].y, xv[q][0].z, xv[q][0].w,
                      xv[q][1].x, xv[q][1].y, xv[q][1].z, xv[q][1].w};
        if (ln) {
          // shifted values of this K range: their sum and sum of squares
          // (the row statistics), and (x - x_0) * g as the operand
          const float g[8] = {gv[q][0].x, gv[q][0].y, gv[q][0].z, gv[q][0].w,
                              gv[q][1].x, gv[q][1].y, gv[q][1].z, gv[q][1].w};
          float s1 = 0.f, s2 = 0.f;
          if (r < Mv) {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float t = f[e] - shv[q];
              s1 += t;
              s2 += t * t;
              f[e] = t * g[e];
            }
          }
          // the eight lanes of one row piece share r
#pragma unroll
          for (int o = 1; o < 8; o <<= 1) {
            s1 += __shfl_xor_sync(0xffffffffu, s1, o);
            s2 += __shfl_xor_sync(0xffffffffu, s2, o);
          }
          if (c == 0 && r < Mv) {
            atomicAdd(&s_s1[r], s1);
            atomicAdd(&s_s2[r], s2);
          }
        }
        uint4 hv, lv;
        __half2* h = reinterpret_cast<__half2*>(&hv);
        __half2* l = reinterpret_cast<__half2*>(&lv);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __half2 hi = __floats2half2_rn(f[2 * e], f[2 * e + 1]);
          const float2 hf = __half22float2(hi);
          h[e] = hi;
          l[e] = __floats2half2_rn(f[2 * e] - hf.x, f[2 * e + 1] - hf.y);
        }
        const int off = j * MT * 128 + r * 128 + ((c ^ (r & 7)) << 4);
        *reinterpret_cast<uint4*>(sXh + off) = hv;
        *reinterpret_cast<uint4*>(sXl + off) = lv;
      }
    }
    fence_async_shared();
    mbar_arrive(x_full);

    // ---- the accumulator: thread = weight row n, TMEM columns = rows m
    // warps 0-3 agree on the outcome before any of them meets barrier 1 again
    if (!mbar_wait_warp(acc_full, 0) && lane == 0) atomicExch(abort_flag, 1);
    named_bar(1, 128);  // also: the statistics of this K range are complete
    ok = *reinterpret_cast<volatile int*>(abort_flag) == 0;
    tc_fence_after_sync();
    const int f = warp * 32 + lane, n = n0 + f;
    const uint32_t taddr = tbase + ((uint32_t)(warp * 32) << 16);
    const float bn = (a.bias && n < a.N) ? __ldg(a.bias + n) : 0.f;
    const int rows = Mv + (ln ? 2 : 0);  // accumulator columns with content
    const float inv_k = 1.0f / (float)a.K;
    if (ok) {
      if (a.S == 1) {
        float cn = 0.f, dn = 0.f;
        if (ln) {
          cn = tmem_ld1(taddr + Mv);
          dn = tmem_ld1(taddr + Mv + 1);
          tmem_wait_ld();
          for (int t = tid; t < Mv; t += 128) lin_row_stats(s_s1[t], s_s2[t], inv_k, a.eps, t, s_dm, s_rs);
          named_bar(1, 128);
        }
        for (int c0 = 0; c0 < Mv; c0 += 16) {
          float v[16];
          tmem_ld16(taddr + c0, v);
          tmem_wait_ld();
          lin_emit16(a, m0 + c0, min(16, Mv - c0), n, v, bn, ln, s_dm + c0, s_rs + c0, cn, dn);
        }
      } else {
        float* accp = a.acc + (int64_t)tile * MT * 128 + f;
        float* stp = a.stats + (int64_t)tile * MT * 2;
        for (int c0 = 0; c0 < rows; c0 += 16) {
          float v[16];
          tmem_ld16(taddr + c0, v);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e)
            if (c0 + e < rows) atomicAdd(accp + (c0 + e) * 128, v[e]);
        }
        if (ln)
          for (int t = tid; t < Mv; t += 128) {
            atomicAdd(stp + 2 * t, s_s1[t]);
            atomicAdd(stp + 2 * t + 1, s_s2[t]);
          }
        __threadfence();
        named_bar(1, 128);
        if (tid == 0) *last_flag = (atomicAdd(&a.tickets[tile], 1u) == (uint32_t)(a.S - 1));
        named_bar(1, 128);
        if (*last_flag) {
          __threadfence();
          float cn = 0.f, dn = 0.f;
          if (ln) {
            cn = __ldcg(accp + Mv * 128);
            dn = __ldcg(accp + (Mv + 1) * 128);
            for (int t = tid; t < Mv; t += 128) {
              const float s1 = __ldcg(stp + 2 * t), s2 = __ldcg(stp + 2 * t + 1);
              lin_row_stats(s1, s2, inv_k, a.eps, t, s_dm, s_rs);
            }
            named_bar(1, 128);
            __stcg(accp + Mv * 128, 0.f);
            __stcg(accp + (Mv + 1) * 128, 0.f);
            for (int t = tid; t < 2 * Mv; t += 128) __stcg(stp + t, 0.f);
          }
          for (int c0 = 0; c0 < Mv; c0 += 16) {
            float v[16];
            const int cnt = min(16, Mv - c0);
#pragma unroll
            for (int e = 0; e < 16; ++e) v[e] = e < cnt ? __ldcg(accp + (c0 + e) * 128) : 0.f;
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (e < cnt) __stcg(accp + (c0 + e) * 128, 0.f);
            lin_emit16(a, m0 + c0, cnt, n, v, bn, ln, s_dm + c0, s_rs + c0, cn, dn);
          }
          if (tid == 0) a.tickets[tile] = 0u;
        }
      }
    }
  }
  if (!ok && lane == 0) set_dev_err(a.dev_err, ASR_DEVERR_TIMEOUT);
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after_sync();
    tmem_dealloc(tbase, a.tmem_cols);
  }
}

struct LinPlan {
  int MT, MR, m_tiles, n_tiles, S, KB, nkb_max;
  uint32_t tmem_cols;
  size_t acc_bytes, stats_bytes, ws_bytes;
  int smem;
};

// Tiles of 128 weight rows x MT operand rows (the sequences of the tile, plus
// the g and b rows with LayerNorm); the K axis split S ways so that the grid
// covers the GPU once without a second wave; the activation planes capped at
// kLinXCap.
static bool lin_plan(int M, int N, int K, bool ln, int sms, LinPlan* p) {
  if (M < 1 || N < 1 || K < 64 || K % 64 != 0 || sms < 1) return false;
  const int extra = ln ? 2 : 0;
  const int per_tile = kLinMaxMT - extra;
  p->m_tiles = (M + per_tile - 1) / per_tile;
  p->MR = (M + p->m_tiles - 1) / p->m_tiles;
  const int mt = p->MR + extra;
  p->MT = mt < 16 ? 16 : (mt + 15) / 16 * 16;
  p->n_tiles = (N + 127) / 128;
  p->KB = K / 64;
  const int tiles = p->m_tiles * p->n_tiles;
  int S = sms / tiles;  // one wave: one CTA per SM at most
  if (S > p->KB) S = p->KB;
  const int cap = kLinXCap / (2 * p->MT * 128);  // k-blocks of activations per CTA (>= 1)
  const int s_min = (p->KB + cap - 1) / cap;
  if (S < s_min) S = s_min;
  if (S < 1) S = 1;
  p->S = S;
  p->nkb_max = (p->KB + S - 1) / S;
  uint32_t cols = 32;
  while (cols < (uint32_t)p->MT) cols <<= 1;
  p->tmem_cols = cols;
  p->acc_bytes = S > 1 ? align_up((size_t)tiles * p->MT * 128 * 4, 256) : 0;
  p->stats_bytes = S > 1 ? align_up((size_t)tiles * p->MT * 2 * 4, 256) : 0;
  p->ws_bytes = S > 1 ? p->acc_bytes + p->stats_bytes + align_up((size_t)tiles * 4, 256) : 0;
  p->smem = kLinSmemFixed + 2 * p->MT * 128 * p->nkb_max;
  return true;
}

static std::once_flag g_lin_attr;

}  // namespace asrkv

using namespace asrkv;

extern "C" size_t asr_linear_workspace_size(int M, int N, int K) {
  LinPlan p, q;  // with and without LayerNorm: the larger serves both
  const int sms = device_sm_count();
  if (!lin_plan(M, N, K, true, sms, &p) || !lin_plan(M, N, K, false, sms, &q)) return 0;
  return p.ws_bytes > q.ws_bytes ? p.ws_bytes : q.ws_bytes;
}

extern "C" int asr_linear(const float* x, int64_t x_stride, const float* ln_g, const float* ln_b,
                          float eps, const uint16_t* w, const float* bias, int M, int N, int K,
                          int mode, float* y, int64_t y_stride, void* ws, size_t ws_bytes,
                          int32_t* dev_err, asr_stream_t stream) {
  if (M < 0 || N < 1 || K < 1 || mode < ASR_LINEAR_STORE || mode > ASR_LINEAR_GELU)
    return ASR_ERR_INVALID_ARG;
  if (K % 64 != 0 || N > (1 << 20) || K > (1 << 20)) return ASR_ERR_UNSUPPORTED;
  if (M == 0) return ASR_OK;
  if (!x || !w || !y || ((ln_g == nullptr) != (ln_b == nullptr))) return ASR_ERR_INVALID_ARG;
  if (x_stride < K || y_stride < N || !(eps >= 0.f)) return ASR_ERR_INVALID_ARG;
  if (!aligned16(x) || x_stride % 4 != 0 || !aligned16(w) ||
      (ln_g && (!aligned16(ln_g) || !aligned16(ln_b))))
    return ASR_ERR_MISALIGNED;
  // y must not overlap x: other CTAs still read x while the epilogue writes y
  const uintptr_t x0 = reinterpret_cast<uintptr_t>(x);
  const uintptr_t x1 = reinterpret_cast<uintptr_t>(x + (int64_t)(M - 1) * x_stride + K);
  const uintptr_t y0 = reinterpret_cast<uintptr_t>(y);
  const uintptr_t y1 = reinterpret_cast<uintptr_t>(y + (int64_t)(M - 1) * y_stride + N);
  if (x0 < y1 && y0 < x1) return ASR_ERR_ALIAS;
  const int sms = device_sm_count();
  if (sms <= 0) return ASR_ERR_CUDA;
  LinPlan p;
  if (!lin_plan(M, N, K, ln_g != nullptr, sms, &p)) return ASR_ERR_UNSUPPORTED;
  if (p.ws_bytes > 0 &&
      (!ws || ws_bytes < p.ws_bytes || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0))
    return ASR_ERR_WORKSPACE;
  static cudaError_t attr = cudaSuccess;
  std::call_once(g_lin_attr, [] {
    attr = cudaFuncSetAttribute(linear_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kLinSmemFixed + kLinXCap);
  });
  if (attr != cudaSuccess) return ASR_ERR_CUDA;
  CUtensorMap tw;
  if (!make_tmap_f16_3d(&tw, w, (uint64_t)K, (uint64_t)N, 1, (uint64_t)K * 2,
                        (uint64_t)N * K * 2, 64, 128))
    return ASR_ERR_CUDA;
  LinArgs la = {};
  la.x = x;
  la.x_stride = x_stride;
  la.ln_g = ln_g;
  la.ln_b = ln_b;
  la.eps = eps;
  la.bias = bias;
  la.y = y;
  la.y_stride = y_stride;
  la.acc = p.S > 1 ? static_cast<float*>(ws) : nullptr;
  unsigned char* wsb = static_cast<unsigned char*>(ws);
  la.stats = p.S > 1 ? reinterpret_cast<float*>(wsb + p.acc_bytes) : nullptr;
  la.tickets =
      p.S > 1 ? reinterpret_cast<uint32_t*>(wsb + p.acc_bytes + p.stats_bytes) : nullptr;
  la.M = M;
  la.N = N;
  la.K = K;
  la.mode = mode;
  la.MT = p.MT;
  la.MR = p.MR;
  la.n_tiles = p.n_tiles;
  la.S = p.S;
  la.KB = p.KB;
  la.nkb_max = p.nkb_max;
  la.tmem_cols = p.tmem_cols;
  la.dev_err = dev_err;
  const int units = p.m_tiles * p.n_tiles * p.S;
  cudaError_t e = launch_pdl(linear_kernel, dim3(units), dim3(kLinThreads), (size_t)p.smem,
                             (cudaStream_t)stream, tw, la);
  return e == cudaSuccess ? ASR_OK : ASR_ERR_CUDA;
}
