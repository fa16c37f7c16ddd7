// linear.cu -- the dense steps of a decoder layer around the attention (next
// row): a pre-norm (LayerNorm or RMSNorm) or a SwiGLU input, then the product
// of the activations with an f16 weight, with a Bias, Residual or Gelu
// epilogue.
//
// Defines: "wavo 0.1.0, src/whisper/decoder.rs", Decoder::record_step
// (layer_norm of x into y; gemv of y with the qkv, self_out, cross_q,
// cross_out, fc1 and fc2 weights, epilogue Bias, Residual(1.0) or Gelu);
// "Nest whisper-tiny, src/lib.linnet", LayerNorm (eps 1e-5) and Mlp (fc2 of
// gelu_erf of fc1); "transcribe.cpp, src/arch/qwen3_asr/decoder.h", header
// comment (pre-norm RMSNorm, SwiGLU MLP down(silu(gate(x)) * up(x))).
//
//   a_m  = LayerNorm(x_m) * g + b  |  RMSNorm(x_m) * g  |  silu(gate_m) * up_m  |  x_m
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
// (N = 1280 is ten tiles) the K axis is split until the grid covers the GPU.
// A residual without a norm is linear in the partial sums, so each CTA adds
// its part straight onto y (red.add).  Otherwise the CTAs of one tile add
// their partial sums into a zero fp32 tile in the workspace with one bulk
// reduction each, and the last to arrive (a counter per tile) loads the sum
// back, applies the epilogue, writes y and puts the tile and the counter
// back to zero.
//
// The norms without a pass over whole rows: a CTA only sees its K range, so
// the normalisation is folded into the product.  LayerNorm: with x_0 the
// row's first element, the operand is (x_k - x_0) * g_k, and two more
// operand rows hold g and b, so the same accumulator collects cn = sum_k g_k
// W_nk and dn = sum_k b_k W_nk; the CTA also sums (x_k - x_0) and its square
// over its K range.  Once all K is in (after the split reduction), mean - x_0
// = s1/K, var = s2/K - (s1/K)^2 and
//   sum_k a_mk W_nk = rstd * (sum_k (x_k - x_0) g_k W_nk - (mean - x_0) cn) + dn.
// Shifting by x_0 keeps both differences of the size of the row's spread.
// RMSNorm: the operand is x_k * g_k, the CTA sums x_k^2, and the sum is
// rstd * sum_k x_k g_k W_nk.  A SwiGLU input forms silu(gate) * up in fp32
// from the two halves of each row while staging.
//
// Roles: warp 8 streams W (128 rows x 64 k per stage, 128-byte swizzle) and
// holds the TMEM allocation; warp 9 issues tcgen05.mma; warps 0-7 bring the
// fp32 activations in with bulk copies and write the hi/lo operand to shared
// memory in the same swizzled layout (with the norm sums); warps 0-3 then
// drain the accumulator (thread = weight row, one TMEM lane each) and run
// the epilogue.  W is never written by a kernel of this library, so the
// weight loads start before the wait on the previous grid (programmatic
// dependent launch): they overlap its tail.
#include <mutex>

#include "common.cuh"
#include "tcgen05.cuh"

namespace asrkv {

constexpr int kLinStages = 4;
constexpr int kLinWTile = 128 * 64 * 2;  // 16 KB: 128 weight rows x 64 k
constexpr int kLinStageThreads = 256;    // warps 0-7 build the operand; warps 0-3 then drain TMEM
constexpr int kLinTmaWarp = 8, kLinMmaWarp = 9;
constexpr int kLinThreads = 320;
constexpr int kLinMaxMT = 256;           // the MMA's N
constexpr int kLinSmemFixed = 1024 + kLinStages * kLinWTile + 256 + 4 * kLinMaxMT * 4;
constexpr int kLinSmemMax = 232448;      // the largest dynamic shared memory of one CTA

// Bytes of the fp32 staging of one CTA: MR rows of its K range (nkb_max
// k-blocks of 64; twice that for a SwiGLU input: gate and up), with a norm
// the same range of its weight, and with LayerNorm also of its bias and 16
// bytes of each row's head.
__host__ __device__ constexpr int lin_f32_bytes(int MR, int nkb_max, int norm, bool glu) {
  return ((MR * (nkb_max * 64 + 4) * (glu ? 2 : 1) +
           (norm != ASR_NORM_NONE ? (nkb_max * 64 + 4) : 0) +
           (norm == ASR_NORM_LAYER ? (nkb_max * 64 + 4) + MR * 4 : 0)) *
              4 +
          15) /
         16 * 16;
}

struct LinArgs {
  const float* x;
  int64_t x_stride;
  const float* norm_w;  // LayerNorm / RMSNorm weight [K] (NULL: no norm)
  const float* norm_b;  // LayerNorm bias [K]
  int norm;             // ASR_NORM_*
  int act;              // ASR_ACT_*
  float eps;
  const float* bias;
  float* y;
  int64_t y_stride;
  float* acc;         // [tiles][MT][128] fp32, zero between calls
  float* stats;       // [tiles][2][MT] fp32 (LayerNorm sums), zero between calls
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

// Bulk (TMA) reduction: global[dst .. dst+bytes) += shared[src ..] as fp32,
// element by element, performed at L2.  16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_reduce_add_f32(float* dst, const float* src, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(
                   dst),
               "r"(smem_addr(src)), "r"(bytes)
               : "memory");
}

// Commit this thread's bulk operations and wait until they have completed
// (their writes performed).
__device__ __forceinline__ void bulk_commit_wait_all() {
  asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group 0;" ::: "memory");
}

// Order this thread's async-proxy accesses of global memory against its
// generic-proxy ones (both directions).
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Row statistics from K-sums.  LayerNorm: of the values shifted by the row's
// first element x_0, s1 = sum (x - x_0), s2 = sum (x - x_0)^2, so dm = mean -
// x_0 and rstd = 1 / sqrt(var + eps), var = s2/K - (s1/K)^2.  RMSNorm: s2 =
// sum x^2, dm = 0 and rstd = 1 / sqrt(s2/K + eps).
__device__ __forceinline__ void lin_row_stats(float s1, float s2, float inv_k, float eps, int t,
                                              float* s_dm, float* s_rs, bool ln) {
  const float dm = ln ? s1 * inv_k : 0.f;  // RMSNorm: the mean square, nothing subtracted
  const float var = fmaxf(s2 * inv_k - dm * dm, 0.f);
  s_dm[t] = dm;
  s_rs[t] = rsqrtf(var + eps);
}

// Old values of a residual's rows m_first .. m_first+cnt-1 at column n, all
// loads issued together (zeros when there is no residual).
__device__ __forceinline__ void lin_load_old(const LinArgs& a, int m_first, int cnt, int n,
                                             bool resid, float* yo) {
  // rows past the last one re-read it (a valid address): no branch per load
#pragma unroll
  for (int e = 0; e < 32; ++e)
    yo[e] = resid ? a.y[(int64_t)(m_first + min(e, cnt - 1)) * a.y_stride + n] : 0.f;
}

// Outputs (m_first + e, n) for e < cnt from the K-sums v[e]:
//   LayerNorm: a_mk = ((x_mk - x_0) - dm) * rstd * g_k + b_k, so
//   sum_k a_mk W_nk = rstd * (v - dm * cn) + dn with cn = sum_k g_k W_nk and
//   dn = sum_k b_k W_nk; RMSNorm: a_mk = x_mk * rstd * g_k, so the sum is
//   rstd * v; otherwise the sum is v itself.  Then bias, epilogue.
__device__ __forceinline__ void lin_emit(const LinArgs& a, int m_first, int cnt, int n,
                                         const float* v, const float* yo, float bn, int norm,
                                         const float* dm, const float* rs, float cn, float dn) {
  if (n >= a.N) return;
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    if (e < cnt) {
      const float t = norm == ASR_NORM_LAYER ? rs[e] * (v[e] - dm[e] * cn) + dn
                      : norm == ASR_NORM_RMS ? rs[e] * v[e]
                                             : v[e];
      a.y[(int64_t)(m_first + e) * a.y_stride + n] = lin_epilogue(a.mode, t + bn, yo[e]);
    }
  }
}

__global__ void __launch_bounds__(kLinThreads, 1)
linear_kernel(const __grid_constant__ CUtensorMap tw, const LinArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int MT = a.MT;
  const bool ln = a.norm == ASR_NORM_LAYER;  // the g and b operand rows, the x_0 shift
  const bool nrm = a.norm != ASR_NORM_NONE;   // row statistics
  const bool glu = a.act == ASR_ACT_SWIGLU;   // activations silu(gate) * up
  const int plane = MT * 128 * a.nkb_max;                  // bytes of one activation plane
  unsigned char* sW = smem;                                // stages x 16 KB
  unsigned char* sXh = sW + kLinStages * kLinWTile;        // hi plane: [nkb][MT rows][128 B]
  unsigned char* sXl = sXh + plane;                        // lo plane
  unsigned char* sFb = sXl + plane;                        // fp32 staging
  const int f32b = lin_f32_bytes(a.MR, a.nkb_max, a.norm, glu);
  uint64_t* full = reinterpret_cast<uint64_t*>(sFb + f32b);
  uint64_t* empty = full + kLinStages;
  uint64_t* xin_full = empty + kLinStages;  // the fp32 activations have landed
  uint64_t* x_full = xin_full + 1;          // the f16 operand is in shared memory
  uint64_t* acc_full = x_full + 1;          // the accumulator is complete
  uint64_t* drain = acc_full + 1;           // every MMA this CTA issued has completed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);
  int* last_flag = reinterpret_cast<int*>(tslot + 1);
  int* abort_flag = last_flag + 1;  // a wait of warps 0-3 gave up
  int* abort_any = abort_flag + 1;  // some wait of this CTA gave up
  float* s_s1 = reinterpret_cast<float*>(sFb + f32b + 256);
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
    mbar_init(xin_full, 1);
    mbar_init(x_full, kLinStageThreads);
    mbar_init(acc_full, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    *abort_any = 0;
    *last_flag = 0;
    fence_barrier_init();
  }
  if (tid < MT) s_s1[tid] = s_s2[tid] = 0.f;
  if (warp == kLinTmaWarp) {
    tmem_alloc(tslot, a.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = *tslot;
  grid_launch_dependents();
  bool ok = true;

  if (warp == kLinTmaWarp) {
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
  } else if (warp == kLinMmaWarp) {
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
    // ================================================ operand (warps 0-7)
    grid_dependency_wait();  // x (and y, the workspace) belong to earlier grids
    // 1. Bulk copies bring this CTA's K range of each activation row (and,
    // with LayerNorm, of g and b, and each row's first 16 bytes) into shared
    // memory as fp32: one round trip.
    const int RS = a.nkb_max * 64 + 4;  // floats per staged row (+4: rows start 16 banks apart)
    float* xs = reinterpret_cast<float*>(sFb);
    float* xu = xs + a.MR * RS;         // SwiGLU: the up half of each row
    float* gs = xu + (glu ? a.MR * RS : 0);
    float* bs = gs + RS;
    float* hs = bs + RS;  // [MR][4]: x_0 of each row in hs[4 r]
    const uint32_t q_bytes = (uint32_t)nkb * 256;
    if (warp == 0) {
      if (lane == 0)
        mbar_arrive_expect_tx(xin_full, Mv * q_bytes * (glu ? 2u : 1u) + (nrm ? q_bytes : 0u) +
                                            (ln ? q_bytes + Mv * 16 : 0u));
      __syncwarp();
      for (int r = lane; r < Mv; r += 32) {
        const float* row = a.x + (int64_t)(m0 + r) * a.x_stride;
        bulk_g2s_plain(xs + r * RS, row + kb0 * 64, q_bytes, xin_full);
        if (glu) bulk_g2s_plain(xu + r * RS, row + a.K + kb0 * 64, q_bytes, xin_full);
        if (ln) bulk_g2s_plain(hs + r * 4, row, 16, xin_full);
      }
      if (nrm && lane == 0) bulk_g2s_plain(gs, a.norm_w + kb0 * 64, q_bytes, xin_full);
      if (ln && lane == 0) bulk_g2s_plain(bs, a.norm_b + kb0 * 64, q_bytes, xin_full);
    }
    if (!mbar_wait(xin_full, 0)) ok = false;
    // 2. The operand: MT rows x nkb k-blocks x eight 16-byte chunks; chunk c
    // of row r sits at c ^ (r % 8) (the 128-byte swizzle the MMA reads).
    // Rows < Mv: the activations (LayerNorm: (x - x_0) * g, see the
    // epilogue); with LayerNorm, row Mv holds g and row Mv+1 holds b, so that
    // the accumulator also collects sum_k g_k W_nk and sum_k b_k W_nk; the
    // rest is zero.  Thread (rr, c) = (tid / 8, tid % 8) converts chunk c of
    // every k-block of rows rr, rr + 32, ... (a warp's four rows are all
    // below MT or all above: MT is a multiple of 16), keeping the row's
    // LayerNorm sums in registers until its last k-block.
    {
      const int rr = tid >> 3, c = tid & 7;
      for (int r = rr; r < MT; r += 32) {
        const float* srow = nullptr;
        if (r < Mv) srow = xs + r * RS;
        else if (ln && r == Mv) srow = gs;
        else if (ln && r == Mv + 1) srow = bs;
        const bool act = nrm && r < Mv;  // a normalised activation row
        const float sh = (ln && r < Mv) ? hs[r * 4] : 0.f;
        float s1 = 0.f, s2 = 0.f;
#pragma unroll 2
        for (int j = 0; j < nkb; ++j) {
          const int ko = j * 64 + c * 8;
          float f[8];
          if (srow) {
            const float4 u0 = *reinterpret_cast<const float4*>(srow + ko);
            const float4 u1 = *reinterpret_cast<const float4*>(srow + ko + 4);
            f[0] = u0.x; f[1] = u0.y; f[2] = u0.z; f[3] = u0.w;
            f[4] = u1.x; f[5] = u1.y; f[6] = u1.z; f[7] = u1.w;
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = 0.f;
          }
          if (glu && r < Mv) {
            // SwiGLU: silu(gate) * up, silu(v) = v / (1 + e^-v)
            const float4 w0 = *reinterpret_cast<const float4*>(xu + r * RS + ko);
            const float4 w1 = *reinterpret_cast<const float4*>(xu + r * RS + ko + 4);
            const float up[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = f[e] / (1.0f + expf(-f[e])) * up[e];
          }
          if (act) {
            // shifted values (LayerNorm; RMSNorm: unshifted): their sum and
            // sum of squares (the row statistics), and (x - x_0) * g as the
            // operand
            const float4 g0 = *reinterpret_cast<const float4*>(gs + ko);
            const float4 g1 = *reinterpret_cast<const float4*>(gs + ko + 4);
            const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float d = f[e] - sh;
              s1 += d;
              s2 += d * d;
              f[e] = d * g[e];
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
        if (nrm) {
          // the eight lanes of one row share r
#pragma unroll
          for (int o = 1; o < 8; o <<= 1) {
            s1 += __shfl_xor_sync(0xffffffffu, s1, o);
            s2 += __shfl_xor_sync(0xffffffffu, s2, o);
          }
          if (c == 0 && act) {
            s_s1[r] = s1;
            s_s2[r] = s2;
          }
        }
      }
    }
    fence_async_shared();
    mbar_arrive(x_full);
    named_bar(1, kLinStageThreads);  // the LayerNorm sums are complete

    if (warp < 4) {
      // ============================================== epilogue (warps 0-3)
      // thread = weight row n (one TMEM lane), TMEM columns = rows m.  The
      // four warps agree on the outcome before any of them meets barrier 2.
      if (!mbar_wait_warp(acc_full, 0) && lane == 0) atomicExch(abort_flag, 1);
      named_bar(2, 128);
      ok = ok && *reinterpret_cast<volatile int*>(abort_flag) == 0;
      tc_fence_after_sync();
      const int f = warp * 32 + lane, n = n0 + f;
      const uint32_t taddr = tbase + ((uint32_t)(warp * 32) << 16);
      const float bn = (a.bias && n < a.N) ? __ldg(a.bias + n) : 0.f;
      const int rows = Mv + (ln ? 2 : 0);  // accumulator columns with content
      const float inv_k = 1.0f / (float)a.K;
      const bool resid = a.mode == ASR_LINEAR_RESIDUAL && n < a.N;
      if (*reinterpret_cast<volatile int*>(abort_flag) == 0) {
        if (a.S == 1) {
          // one CTA holds the whole K of its tile (the plan splits K at
          // least twice under a norm, so there is no norm here)
          const float cn = 0.f, dn = 0.f;
          for (int c0 = 0; c0 < Mv; c0 += 32) {
            const int cnt = min(32, Mv - c0);
            float v[32], yo[32];
            tmem_ld16(taddr + c0, v);
            if (c0 + 16 < MT) tmem_ld16(taddr + c0 + 16, v + 16);  // MT is a multiple of 16
            lin_load_old(a, m0 + c0, cnt, n, resid, yo);
            tmem_wait_ld();
            lin_emit(a, m0 + c0, cnt, n, v, yo, bn, a.norm, s_dm + c0, s_rs + c0, cn, dn);
          }
        } else if (a.mode == ASR_LINEAR_RESIDUAL && !nrm) {
          // a residual without LayerNorm is linear in each partial sum: every
          // K split adds its part (split 0 with the bias) straight onto y
          const float b0 = s == 0 ? bn : 0.f;
          for (int c0 = 0; c0 < Mv; c0 += 16) {
            float v[16];
            tmem_ld16(taddr + c0, v);
            tmem_wait_ld();
            if (n < a.N) {
#pragma unroll
              for (int e = 0; e < 16; ++e)
                if (c0 + e < Mv) atomicAdd(a.y + (int64_t)(m0 + c0 + e) * a.y_stride + n, v[e] + b0);
            }
          }
        } else if (rows <= 128) {
          // Split K, one pass of bulk operations: the partial tile goes
          // through shared memory (the W ring, free now) and is added into
          // the workspace tile with one bulk reduction; the last CTA of the
          // tile loads the whole sum back with one bulk copy.
          float* P = reinterpret_cast<float*>(sW);  // [rows][128] fp32
          float* acct = a.acc + (int64_t)tile * MT * 128;
          float* stt = a.stats + (int64_t)tile * MT * 2;
          for (int c0 = 0; c0 < rows; c0 += 16) {
            float v[16];
            tmem_ld16(taddr + c0, v);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (c0 + e < rows) P[(c0 + e) * 128 + f] = v[e];
          }
          fence_async_shared();
          named_bar(2, 128);
          if (tid == 0) {
            bulk_reduce_add_f32(acct, P, (uint32_t)rows * 512);
            if (nrm) {
              bulk_reduce_add_f32(stt, s_s1, (uint32_t)MT * 4);
              bulk_reduce_add_f32(stt + MT, s_s2, (uint32_t)MT * 4);
            }
            bulk_commit_wait_all();     // the sums are in global memory
            fence_proxy_async_global();  // ... and ordered before the ticket
            __threadfence();
            *last_flag = (atomicAdd(&a.tickets[tile], 1u) == (uint32_t)(a.S - 1));
            if (*last_flag) {
              __threadfence();
              fence_proxy_async_global();
              mbar_arrive_expect_tx(xin_full, (uint32_t)rows * 512 + (nrm ? (uint32_t)MT * 8 : 0u));
              bulk_g2s_plain(P, acct, (uint32_t)rows * 512, xin_full);
              if (nrm) {
                bulk_g2s_plain(s_s1, stt, (uint32_t)MT * 4, xin_full);
                bulk_g2s_plain(s_s2, stt + MT, (uint32_t)MT * 4, xin_full);
              }
            }
          }
          named_bar(2, 128);
          if (*last_flag) {
            // xin_full's second phase: the whole tile and its row sums
            if (!mbar_wait(xin_full, 1)) atomicExch(abort_flag, 1);
            float cn = 0.f, dn = 0.f;
            if (ln) {
              cn = P[Mv * 128 + f];
              dn = P[(Mv + 1) * 128 + f];
            }
            if (nrm)
              for (int t = tid; t < Mv; t += 128)
                lin_row_stats(s_s1[t], s_s2[t], inv_k, a.eps, t, s_dm, s_rs, ln);
            named_bar(2, 128);
            // put the workspace back to zero
            for (int m = 0; m < rows; ++m) __stcg(acct + m * 128 + f, 0.f);
            if (nrm)
              for (int t = tid; t < 2 * MT; t += 128) __stcg(stt + t, 0.f);
            if (tid == 0) a.tickets[tile] = 0u;
            for (int c0 = 0; c0 < Mv; c0 += 32) {
              const int cnt = min(32, Mv - c0);
              float v[32], yo[32];
              lin_load_old(a, m0 + c0, cnt, n, resid, yo);
#pragma unroll
              for (int e = 0; e < 32; ++e) v[e] = P[min(c0 + e, rows - 1) * 128 + f];
              lin_emit(a, m0 + c0, cnt, n, v, yo, bn, a.norm, s_dm + c0, s_rs + c0, cn, dn);
            }
            if (*reinterpret_cast<volatile int*>(abort_flag) != 0) ok = false;
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
          if (nrm)
            for (int t = tid; t < Mv; t += 128) {
              atomicAdd(stp + t, s_s1[t]);
              atomicAdd(stp + MT + t, s_s2[t]);
            }
          __threadfence();
          named_bar(2, 128);
          if (tid == 0) *last_flag = (atomicAdd(&a.tickets[tile], 1u) == (uint32_t)(a.S - 1));
          named_bar(2, 128);
          if (*last_flag) {
            __threadfence();
            float cn = 0.f, dn = 0.f;
            for (int c0 = 0; c0 < Mv; c0 += 32) {
              const int cnt = min(32, Mv - c0);
              float v[32], yo[32];
              // every load of the chunk is issued before any is used; rows
              // past the tile re-read its last row (always a valid address)
#pragma unroll
              for (int e = 0; e < 32; ++e) v[e] = __ldcg(accp + min(c0 + e, MT - 1) * 128);
              lin_load_old(a, m0 + c0, cnt, n, resid, yo);
              if (c0 == 0 && nrm) {
                if (ln) {
                  cn = __ldcg(accp + Mv * 128);
                  dn = __ldcg(accp + (Mv + 1) * 128);
                }
                for (int t = tid; t < Mv; t += 128)
                  lin_row_stats(__ldcg(stp + t), __ldcg(stp + MT + t), inv_k, a.eps, t, s_dm,
                                s_rs, ln);
                named_bar(2, 128);  // uniform: every thread of the last CTA is here
                if (ln) {
                  __stcg(accp + Mv * 128, 0.f);
                  __stcg(accp + (Mv + 1) * 128, 0.f);
                }
                for (int t = tid; t < Mv; t += 128) {
                  __stcg(stp + t, 0.f);
                  __stcg(stp + MT + t, 0.f);
                }
              }
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (e < cnt) __stcg(accp + (c0 + e) * 128, 0.f);
              lin_emit(a, m0 + c0, cnt, n, v, yo, bn, a.norm, s_dm + c0, s_rs + c0, cn, dn);
            }
            if (tid == 0) a.tickets[tile] = 0u;
          }
        }
      } else {
        ok = false;
      }
    }
  }
  if (!ok && lane == 0) {
    set_dev_err(a.dev_err, ASR_DEVERR_TIMEOUT);
    atomicExch(abort_any, 1);
  }
  tc_fence_before_sync();
  __syncthreads();
  // After a wait gave up, nothing may still be in flight into this CTA's
  // shared memory or tensor memory when it frees them and leaves: the bulk
  // copies of warp 0 into xin_full (the activations, its first phase, and in
  // the last CTA of a tile the reloaded sums, its second; bounded waits; the
  // W producer already waited for its own copies above) and every MMA the
  // MMA warp issued (a commit tracks all of them).
  if (*reinterpret_cast<volatile int*>(abort_any)) {
    if (warp == 0) {
      mbar_wait_warp(xin_full, *reinterpret_cast<volatile int*>(last_flag) ? 1 : 0);
    } else if (warp == kLinMmaWarp) {
      mma_commit_warp(drain);
      mbar_wait_warp(drain, 0);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kLinTmaWarp) {
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
// covers the GPU once without a second wave, more if one CTA's share of the
// activations would not fit in shared memory.
static bool lin_plan(int M, int N, int K, int norm, bool glu, int sms, LinPlan* p) {
  if (M < 1 || N < 1 || K < 64 || K % 64 != 0 || sms < 1) return false;
  const int extra = norm == ASR_NORM_LAYER ? 2 : 0;
  const int per_tile = kLinMaxMT - extra;
  p->n_tiles = (N + 127) / 128;
  p->KB = K / 64;
  // under a norm the K axis is always split (the norm terms are applied by
  // the last CTA of a tile, after the split reduction)
  const int s_min = norm != ASR_NORM_NONE ? 2 : 1;
  if (p->KB < s_min) return false;
  // more, shorter row tiles when even one k-block of a tile's activations
  // would not fit in shared memory (wide SwiGLU rows)
  for (p->m_tiles = (M + per_tile - 1) / per_tile; p->m_tiles <= M; ++p->m_tiles) {
    p->MR = (M + p->m_tiles - 1) / p->m_tiles;
    const int mt = p->MR + extra;
    p->MT = mt < 16 ? 16 : (mt + 15) / 16 * 16;
    const int tiles = p->m_tiles * p->n_tiles;
    int S = sms / tiles;  // one wave: one CTA per SM at most
    if (S > p->KB) S = p->KB;
    if (S < s_min) S = s_min;
    auto smem_of = [&](int s) {
      const int nkb = (p->KB + s - 1) / s;
      return kLinSmemFixed + 2 * p->MT * 128 * nkb + lin_f32_bytes(p->MR, nkb, norm, glu);
    };
    while (smem_of(S) > kLinSmemMax && S < p->KB) ++S;  // fewer k-blocks per CTA
    if (smem_of(S) > kLinSmemMax) continue;
    p->S = S;
    p->nkb_max = (p->KB + S - 1) / S;
    uint32_t cols = 32;
    while (cols < (uint32_t)p->MT) cols <<= 1;
    p->tmem_cols = cols;
    p->acc_bytes = S > 1 ? align_up((size_t)tiles * p->MT * 128 * 4, 256) : 0;
    p->stats_bytes = S > 1 ? align_up((size_t)tiles * p->MT * 2 * 4, 256) : 0;
    p->ws_bytes = S > 1 ? p->acc_bytes + p->stats_bytes + align_up((size_t)tiles * 4, 256) : 0;
    p->smem = smem_of(S);
    return true;
  }
  return false;
}

}  // namespace asrkv

using namespace asrkv;

extern "C" size_t asr_linear_workspace_size(int M, int N, int K) {
  // the largest over the norms and inputs: one workspace serves every call
  const int sms = device_sm_count();
  const int cases[4][2] = {{ASR_NORM_NONE, 0}, {ASR_NORM_LAYER, 0}, {ASR_NORM_RMS, 0},
                           {ASR_NORM_NONE, 1}};
  size_t best = 0;
  for (const auto& c : cases) {
    LinPlan p;
    if (lin_plan(M, N, K, c[0], c[1] != 0, sms, &p) && p.ws_bytes > best) best = p.ws_bytes;
  }
  return best;
}

extern "C" int asr_linear(const float* x, int64_t x_stride, int norm, const float* norm_w,
                          const float* norm_b, float eps, int act, const uint16_t* w,
                          const float* bias, int M, int N, int K, int mode, float* y,
                          int64_t y_stride, void* ws, size_t ws_bytes, int32_t* dev_err,
                          asr_stream_t stream) {
  if (M < 0 || N < 1 || K < 1 || mode < ASR_LINEAR_STORE || mode > ASR_LINEAR_GELU ||
      norm < ASR_NORM_NONE || norm > ASR_NORM_RMS || act < ASR_ACT_NONE || act > ASR_ACT_SWIGLU)
    return ASR_ERR_INVALID_ARG;
  if (K % 64 != 0 || N > (1 << 20) || K > (1 << 20)) return ASR_ERR_UNSUPPORTED;
  if (act == ASR_ACT_SWIGLU && norm != ASR_NORM_NONE) return ASR_ERR_UNSUPPORTED;
  if (norm != ASR_NORM_NONE && K < 128) return ASR_ERR_UNSUPPORTED;
  if (M == 0) return ASR_OK;
  const int xw = act == ASR_ACT_SWIGLU ? 2 * K : K;  // x values read per row
  if (!x || !w || !y) return ASR_ERR_INVALID_ARG;
  if ((norm != ASR_NORM_NONE && !norm_w) || (norm == ASR_NORM_LAYER && !norm_b))
    return ASR_ERR_INVALID_ARG;
  if (x_stride < xw || y_stride < N || !(eps >= 0.f)) return ASR_ERR_INVALID_ARG;
  if (!aligned16(x) || x_stride % 4 != 0 || !aligned16(w) ||
      (norm != ASR_NORM_NONE && !aligned16(norm_w)) ||
      (norm == ASR_NORM_LAYER && !aligned16(norm_b)))
    return ASR_ERR_MISALIGNED;
  // y must not overlap x: other CTAs still read x while the epilogue writes y
  const uintptr_t x0 = reinterpret_cast<uintptr_t>(x);
  const uintptr_t x1 = reinterpret_cast<uintptr_t>(x + (int64_t)(M - 1) * x_stride + xw);
  const uintptr_t y0 = reinterpret_cast<uintptr_t>(y);
  const uintptr_t y1 = reinterpret_cast<uintptr_t>(y + (int64_t)(M - 1) * y_stride + N);
  if (x0 < y1 && y0 < x1) return ASR_ERR_ALIAS;
  const int sms = device_sm_count();
  if (sms <= 0) return ASR_ERR_CUDA;
  LinPlan p;
  if (!lin_plan(M, N, K, norm, act == ASR_ACT_SWIGLU, sms, &p)) return ASR_ERR_UNSUPPORTED;
  if (p.ws_bytes > 0 &&
      (!ws || ws_bytes < p.ws_bytes || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0))
    return ASR_ERR_WORKSPACE;
  if (ensure_dynamic_smem((const void*)linear_kernel, kLinSmemMax) != cudaSuccess)
    return ASR_ERR_CUDA;
  CUtensorMap tw;
  if (!make_tmap_f16_3d(&tw, w, (uint64_t)K, (uint64_t)N, 1, (uint64_t)K * 2,
                        (uint64_t)N * K * 2, 64, 128))
    return ASR_ERR_CUDA;
  LinArgs la = {};
  la.x = x;
  la.x_stride = x_stride;
  la.norm_w = norm != ASR_NORM_NONE ? norm_w : nullptr;
  la.norm_b = norm == ASR_NORM_LAYER ? norm_b : nullptr;
  la.norm = norm;
  la.act = act;
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
