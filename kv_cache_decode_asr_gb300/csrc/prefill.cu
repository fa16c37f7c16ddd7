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
// a8 attention (5th-generation tensor cores): one CTA per (pair of adjacent
//   128-query tiles, sequence, query head), warp-specialised.  Q, K and V^T tiles
//   arrive by tiled TMA with the 128-byte swizzle; S = Q K^T (128 x 64 per
//   key tile) and O += P V are tcgen05.mma kind::f16 (f16 operands, fp32
//   accumulators in tensor memory).  Two softmax groups of 256 threads (one
//   per query tile, two threads per query row, each on half of the 64 key
//   columns) read S from TMEM, run the online softmax
//   in fp32 (log2 domain), rescale O in TMEM only when a row maximum grows by
//   more than 2^8 (the normalisation at the end is exact either way), and
//   write P (f16) back into tensor memory over its S buffer, where the PV MMA
//   reads it as its A operand; S/P are double-buffered, so the tensor core
//   works on one tile while the other is softmaxed.
//   Only key tiles at or below the diagonal are visited (causal).
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
  const int tid = threadIdx.x;
  const int b = blockIdx.y;
  const int t0 = blockIdx.x * kPrepT;
  const int kw = a.Hkv * HD;
  grid_launch_dependents();
  grid_dependency_wait();

  // V rows of the chunk: every load is issued now, so their latency overlaps
  // the rotation table below (kPrepV 16-byte vectors per thread)
  constexpr int kPrepV = 8;
  const int vec_per_row = kw / 8;
  const int nv = kPrepT * vec_per_row;
  uint4 vval[kPrepV];
#pragma unroll
  for (int u = 0; u < kPrepV; ++u) {
    const int idx = tid + u * (int)blockDim.x;
    const int tt = idx / vec_per_row, c = idx % vec_per_row;
    vval[u] = make_uint4(0u, 0u, 0u, 0u);
    if (idx < nv && t0 + tt < a.T)
      vval[u] = *reinterpret_cast<const uint4*>(a.v + ((int64_t)b * a.T + t0 + tt) * kw + c * 8);
  }

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
  // V rows: to the cache, and staged for the transpose
#pragma unroll
  for (int u = 0; u < kPrepV; ++u) {
    const int idx = tid + u * (int)blockDim.x;
    if (idx < nv) {
      const int tt = idx / vec_per_row, c = idx % vec_per_row;
      if (t0 + tt < a.T)
        *reinterpret_cast<uint4*>(a.cache + (int64_t)b * a.seq_stride + (int64_t)(t0 + tt) * 2 * kw +
                                  kw + c * 8) = vval[u];
      *reinterpret_cast<uint4*>(vsm + tt * kw + c * 8) = vval[u];
    }
  }
  // the rows past the first blockDim * kPrepV vectors (more KV heads than
  // the registers cover) go the plain way
  for (int idx = tid + kPrepV * (int)blockDim.x; idx < nv; idx += blockDim.x) {
    const int tt = idx / vec_per_row, c = idx % vec_per_row;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (t0 + tt < a.T) {
      val = *reinterpret_cast<const uint4*>(a.v + ((int64_t)b * a.T + t0 + tt) * kw + c * 8);
      *reinterpret_cast<uint4*>(a.cache + (int64_t)b * a.seq_stride + (int64_t)(t0 + tt) * 2 * kw +
                                kw + c * 8) = val;
    }
    *reinterpret_cast<uint4*>(vsm + tt * kw + c * 8) = val;
  }
  __syncthreads();

  // normed + roped heads: a half-warp per (position, head) vector; lane hl
  // of the half-warp holds dims 8*hl .. 8*hl+7, so lanes hl and hl ^ 8 hold
  // NeoX RoPE partners (i, i + 64).  Each half-warp loads kPrepU vectors
  // before reducing any of them, so several 16-byte loads per lane are in
  // flight.
  constexpr int kPrepU = 4;
  const int hw = tid >> 4, hl = tid & 15;
  const bool upper = hl >= 8;
  const int ib = (hl & 7) * 8;  // frequency index of this lane's first dim
  float wqr[8], wkr[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    wqr[e] = a.wq[8 * hl + e];
    wkr[e] = a.wk[8 * hl + e];
  }
  const int nheads = a.Hq + a.Hkv;
  const int items = kPrepT * nheads;
  const int n_hw = blockDim.x >> 4;
  for (int base = hw; base < items; base += n_hw * kPrepU) {
    uint4 x[kPrepU];
    const uint16_t* srcs[kPrepU];
#pragma unroll
    for (int u = 0; u < kPrepU; ++u) {
      const int item = base + n_hw * u;
      const int tt = item / nheads, hh = item % nheads, t = t0 + tt;
      x[u] = make_uint4(0u, 0u, 0u, 0u);
      srcs[u] = nullptr;
      if (item < items && t < a.T) {
        srcs[u] = hh < a.Hq ? a.q + ((int64_t)b * a.T + t) * a.Hq * HD + hh * HD
                            : a.k + ((int64_t)b * a.T + t) * kw + (hh - a.Hq) * HD;
        x[u] = *reinterpret_cast<const uint4*>(srcs[u] + 8 * hl);
      }
    }
#pragma unroll
    for (int u = 0; u < kPrepU; ++u) {
      // every lane runs the shuffles (both half-warps of a warp stay converged)
      const int item = base + n_hw * u;
      const int tt = min(item / nheads, kPrepT - 1), hh = item % nheads, t = t0 + tt;
      const bool is_q = hh < a.Hq;
      float f[8];
      h8_to_f8(x[u], f);
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float rinv = 1.0f / sqrtf(ss / (float)HD + a.eps);
      float xn[8], y[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) xn[e] = (is_q ? wqr[e] : wkr[e]) * (f[e] * rinv);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float pe = __shfl_xor_sync(0xffffffffu, xn[e], 8);
        const float c = cs[tt * HALF + ib + e], sv = sn[tt * HALF + ib + e];
        y[e] = upper ? xn[e] * c + pe * sv : xn[e] * c - pe * sv;
      }
      if (srcs[u] != nullptr) {
        uint16_t* dst = is_q ? a.qhat + (((int64_t)b * a.T + t) * a.Hq + hh) * HD
                             : a.cache + (int64_t)b * a.seq_stride + (int64_t)t * 2 * kw +
                                   (hh - a.Hq) * HD;
        *reinterpret_cast<uint4*>(dst + 8 * hl) = f8_to_h8(y);
      }
    }
  }

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
  int B, T, Hq, Hkv, n_qt, n_pairs, n_items;
  float sl2e;   // scale * log2(e)
  float* out;   // [B][T][Hq*128] fp32
  int32_t* dev_err;
};

constexpr int kQTile = 128 * 128 * 2;     // 128 queries x 128 dims, f16
constexpr int kKTile = 64 * 128 * 2;      // 64 keys x 128 dims
constexpr int kVTile = 128 * 64 * 2;      // V^T: 128 dims x 64 keys
constexpr int kKVStages = 4;
constexpr int kBarBytes = 1024;           // mbarriers and the TMEM address
constexpr int kXchBytes = 6 * 1024;       // row maxima [tile parity][slot][half][128], row sums [slot][half][128]
constexpr int kAttnSmem = 2 * kQTile + kKVStages * (kKTile + kVTile) + kBarBytes + kXchBytes + 1024;
constexpr int kAttnThreads = 576;  // warps 0-7, 8-15: softmax of slots A, B; 16: TMA; 17: MMA
constexpr float kRescaleLog2 = 8.0f;      // rescale O only when the row max grows by > 2^8

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One work item: two adjacent query tiles of one (sequence, head), tile A =
// 2p in slot A and tile B = 2p+1 in slot B (a lone last tile when n_qt is
// odd).  Their causal lengths differ by one 128-key tile, so both softmax
// groups stay busy side by side on the same K/V stream.
struct PfItem {
  int b, h, kvh, qt_a, qt_b, nA, nB, n;
};

__device__ __forceinline__ PfItem pf_item(const PrefillAttnArgs& a, int it) {
  const int BH = a.B * a.Hq;
  const int pair = a.n_pairs - 1 - it / BH;  // items run longest pairs first
  const int bh = it % BH;
  PfItem x;
  x.b = bh / a.Hq;
  x.h = bh % a.Hq;
  x.kvh = x.h / (a.Hq / a.Hkv);
  x.qt_a = 2 * pair;
  x.qt_b = 2 * pair + 1;
  x.nA = 2 * (x.qt_a + 1);  // 64-key tiles up to the tile's last row (causal)
  x.nB = x.qt_b < a.n_qt ? 2 * (x.qt_b + 1) : 0;
  x.n = x.nA > x.nB ? x.nA : x.nB;
  return x;
}

// The k-th item of this CTA, or -1: rounds of gridDim.x items in snake order
// (even rounds left to right, odd rounds right to left), which with items
// sorted by length spreads the work evenly over the persistent CTAs.
__device__ __forceinline__ int pf_item_index(int k, int n_items) {
  const int P = (int)gridDim.x, c = (int)blockIdx.x;
  const int it = k * P + ((k & 1) ? P - 1 - c : c);
  return it < n_items ? it : -1;
}

// Persistent: one CTA per SM walks its items (pf_item_index) with three
// roles.  Warps 0-7 and 8-15 run the softmax of slots A and B, two threads
// per query row (warp w reads TMEM lanes 32*(w%4)..+31; warps w and w+4 take
// the two halves of the row's keys and of its O columns and exchange their
// partial row maxima through shared memory).  Warp 16 owns the TMEM
// allocation and issues the TMA loads (Q per item, K and V^T per 64-key tile
// through a ring that runs on across items).  Warp 17 issues the MMAs.  Every
// barrier's phase is counted across items, so the next item's Q and K/V
// loads and its first S products overlap the end of the current item, and
// its first PV waits only until the softmax has read the previous O.
// Launched with kAttnThreads threads; prefill.cu is compiled with a register
// cap (build.py) that keeps kAttnThreads x registers within one SM's file.
__global__ void prefill_attn_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                        const __grid_constant__ CUtensorMap tv, const PrefillAttnArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  unsigned char* sQ = smem;                                  // [A, B] x 32 KB
  unsigned char* sK = sQ + 2 * kQTile;                       // stages x 16 KB
  unsigned char* sV = sK + kKVStages * kKTile;               // stages x 16 KB
  uint64_t* bar = reinterpret_cast<uint64_t*>(sV + kKVStages * kVTile);
  uint64_t* q_full = bar;                   // 1: Q of the item landed
  uint64_t* q_empty = q_full + 1;           // 1: the item's S products are done with Q
  uint64_t* kv_full = q_empty + 1;          // kKVStages
  uint64_t* kv_empty = kv_full + kKVStages;
  uint64_t* s_full = kv_empty + kKVStages;  // [A0, A1, B0, B1]: S of slot i, buffer g % 2
  uint64_t* p_full = s_full + 4;            // [A0, A1, B0, B1]: P of slot i, buffer g % 2
  uint64_t* o_done = p_full + 4;            // [A0, A1, B0, B1]: PV of slot tile g -> g % 2
  uint64_t* o_free = o_done + 4;            // [A, B]: the softmax has read O of its item
  uint64_t* xbar = o_free + 2;              // [A, B]: exchange between the two row halves
  uint32_t* tslot = reinterpret_cast<uint32_t*>(xbar + 2);
  float* xmax = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(bar) + kBarBytes);
  float* xsum = xmax + 2 * 2 * 2 * 128;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < kKVStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[i], 8);  // one arrival per softmax warp of the slot
      mbar_init(&o_done[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&o_free[i], 8);
      mbar_init(&xbar[i], 8);
    }
    fence_barrier_init();
  }
  if (warp == 16) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  grid_launch_dependents();
  grid_dependency_wait();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = *tslot;
  // TMEM columns: S of slot i, buffer u at 64*(2i+u) (0..255), O_A 256..383,
  // O_B 384..511.  S is double-buffered so the tensor core computes S(g+1)
  // while the softmax works on S(g).
  auto tS = [&](int i, int u) { return tbase + 64u * (2 * i + u); };
  auto tO = [&](int i) { return tbase + 256u + 128u * i; };

  if (warp == 16) {
    // ======================================================= TMA producer
    // The whole warp runs the schedule; one elected lane issues each copy.
    int gk = 0;  // K/V tiles loaded so far (ring position)
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int it = pf_item_index(k, a.n_items);
      if (it < 0) break;
      const PfItem x = pf_item(a, it);
      // Q is overwritten once the previous item's S products are done
      if (k > 0 && !(ok = mbar_wait_warp(q_empty, (k - 1) & 1))) break;
      mbar_arrive_expect_tx_warp(q_full, x.nB > 0 ? 2 * kQTile : kQTile);
      tma_load_3d_warp(sQ, &tq, x.h * 128, x.qt_a * 128, x.b, q_full);
      tma_load_3d_warp(sQ + kQTile / 2, &tq, x.h * 128 + 64, x.qt_a * 128, x.b, q_full);
      if (x.nB > 0) {
        tma_load_3d_warp(sQ + kQTile, &tq, x.h * 128, x.qt_b * 128, x.b, q_full);
        tma_load_3d_warp(sQ + kQTile + kQTile / 2, &tq, x.h * 128 + 64, x.qt_b * 128, x.b, q_full);
      }
      for (int j = 0; j < x.n; ++j, ++gk) {
        const int s = gk % kKVStages;
        if (gk >= kKVStages && !(ok = mbar_wait_warp(&kv_empty[s], ((gk / kKVStages) - 1) & 1)))
          break;
        mbar_arrive_expect_tx_warp(&kv_full[s], kKTile + kVTile);
        tma_load_3d_warp(sK + s * kKTile, &tk, x.kvh * 128, j * 64, x.b, &kv_full[s]);
        tma_load_3d_warp(sK + s * kKTile + kKTile / 2, &tk, x.kvh * 128 + 64, j * 64, x.b,
                         &kv_full[s]);
        tma_load_3d_warp(sV + s * kVTile, &tv, j * 64, 0, x.b * a.Hkv + x.kvh, &kv_full[s]);
      }
    }
    if (!ok && lane == 0) set_dev_err(a.dev_err, ASR_DEVERR_TIMEOUT);
  } else if (warp == 17) {
    // ======================================================= MMA issuer
    // The whole warp runs the schedule (operand descriptors stay
    // warp-uniform); one elected lane issues each tcgen05 operation.
    constexpr uint32_t kIdS = mma_idesc_f16_f32(128, 64);    // S = Q K^T: 128 x 64
    constexpr uint32_t kIdO = mma_idesc_f16_f32(128, 128);   // O += P V: 128 x 128
    const uint32_t aQ = smem_addr(sQ), aK = smem_addr(sK), aV = smem_addr(sV);
    int gk = 0;             // K/V tiles consumed so far
    int gx[2] = {0, 0};     // tiles of slot A / B so far (S, P and PV barrier phases)
    int ox[2] = {0, 0};     // items whose O slot A / B has accumulated so far
    bool ok = true;
    for (int k = 0; ok; ++k) {
      const int it = pf_item_index(k, a.n_items);
      if (it < 0) break;
      const PfItem x = pf_item(a, it);
      const int nX[2] = {x.nA, x.nB};
      ok = mbar_wait_warp(q_full, k & 1) &&
           mbar_wait_warp(&kv_full[gk % kKVStages], (gk / kKVStages) & 1);
      if (!ok) break;
      tc_fence_after_sync();
      int s_left = x.nA + x.nB;  // S products of this item still to issue
      // S(g) of slot i goes to buffer g % 2; that buffer's previous P (tile
      // g-2) was consumed by a PV issued before this S
      auto issue_s = [&](int i, int j) {
        const int st = (gk + j) % kKVStages;
        const int g = gx[i] + j;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * (kQTile / 2) + (kk & 3) * 32;
          const uint32_t koff = (kk >> 2) * (kKTile / 2) + (kk & 3) * 32;
          mma_f16_warp(tS(i, g & 1), sw128_kmajor_desc(aQ + i * kQTile + off),
                       sw128_kmajor_desc(aK + st * kKTile + koff), kIdS, kk > 0);
        }
        mma_commit_warp(&s_full[2 * i + (g & 1)]);
        if (--s_left == 0) mma_commit_warp(q_empty);  // Q free once these finish
      };
      // P(g) sits in TMEM over its S buffer: 64 keys packed two per column
      auto issue_pv = [&](int i, int j) {
        const int st = (gk + j) % kKVStages;
        const int g = gx[i] + j;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f16_ts_warp(tO(i), tS(i, g & 1) + kk * 8,
                          sw128_kmajor_desc(aV + st * kVTile + kk * 32), kIdO,
                          (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit_warp(&o_done[2 * i + (g & 1)]);
      };
      // S runs two tiles ahead of PV within each slot
      issue_s(0, 0);
      if (x.nB > 0) issue_s(1, 0);
      if (x.n > 1) {
        ok = mbar_wait_warp(&kv_full[(gk + 1) % kKVStages], ((gk + 1) / kKVStages) & 1);
        tc_fence_after_sync();
        if (ok && 1 < x.nA) issue_s(0, 1);
        if (ok && 1 < x.nB) issue_s(1, 1);
      }
      for (int j = 0; j < x.n && ok; ++j) {
        if (j + 2 < x.n) {
          ok = mbar_wait_warp(&kv_full[(gk + j + 2) % kKVStages], ((gk + j + 2) / kKVStages) & 1);
          tc_fence_after_sync();
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (ok && j < nX[i]) {
            const int g = gx[i] + j;
            ok = mbar_wait_warp(&p_full[2 * i + (g & 1)], (g >> 1) & 1);
            // the first PV of an item overwrites O: the softmax must have
            // read the previous item's O first
            if (ok && j == 0 && ox[i] > 0) ok = mbar_wait_warp(&o_free[i], (ox[i] - 1) & 1);
            tc_fence_after_sync();
            if (ok) issue_pv(i, j);
            if (i == 0 && ok && j + 2 < x.nA) issue_s(0, j + 2);
          }
        }
        mma_commit_warp(&kv_empty[(gk + j) % kKVStages]);  // stage free once these finish
        if (ok && j + 2 < x.nB) issue_s(1, j + 2);
      }
      gx[0] += x.nA;
      gx[1] += x.nB;
      ox[0] += x.nA > 0 ? 1 : 0;
      ox[1] += x.nB > 0 ? 1 : 0;
      gk += x.n;
    }
    if (!ok && lane == 0) set_dev_err(a.dev_err, ASR_DEVERR_TIMEOUT);
  } else {
    // ======================================================= softmax
    const int i = warp >> 3;                  // 0: slot A, 1: slot B
    const int hh = (warp >> 2) & 1;           // which half of the keys / O columns
    const int row = (warp & 3) * 32 + lane;   // 0..127: TMEM lane = query row
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    // The two halves of a row meet through xbar[i] (8 warps, one arrival
    // each); xe counts its completed phases.  All waits are warp-uniform and
    // bounded, so a timeout ends every role's loop instead of stranding a
    // warp at a barrier.
    int xe = 0;
    auto exchange = [&]() -> bool {
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&xbar[i]);
      const bool r = mbar_wait_warp(&xbar[i], xe & 1);
      ++xe;
      tc_fence_after_sync();
      return r;
    };
    int g = 0;  // tiles of this slot so far
    bool ok = true;
    float v[32];
    for (int k = 0; ok; ++k) {
      const int it = pf_item_index(k, a.n_items);
      if (it < 0) break;
      const PfItem x = pf_item(a, it);
      const int ni = i == 0 ? x.nA : x.nB;
      if (ni == 0) continue;
      const int q0 = (i == 0 ? x.qt_a : x.qt_b) * 128;
      const int qidx = q0 + row;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < ni && ok; ++j, ++g) {
        ok = mbar_wait_warp(&s_full[2 * i + (g & 1)], (g >> 1) & 1);
        if (!ok) break;
        tc_fence_after_sync();
        tmem_ld32(tS(i, g & 1) + lane_off + 32 * hh, v);
        tmem_wait_ld();
        const int key0 = j * 64 + 32 * hh;
        if (key0 + 31 > q0) {  // some keys of this half lie past some rows
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (key0 + c > qidx) v[c] = -INFINITY;
        }
        float mx[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx[e] = fmaxf(fmaxf(v[e], v[e + 8]), fmaxf(v[e + 16], v[e + 24]));
        const float pmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                 fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        // the row max needs both halves; the exchange also orders both
        // halves' TMEM reads of S before either overwrites part of it with P.
        // Buffers alternate with the tile, so a half never overwrites a value
        // its partner has yet to read.
        float* xb = xmax + ((g & 1) * 2 + i) * 256;
        xb[hh * 128 + row] = pmax;
        ok = exchange();
        if (!ok) break;
        const float tmax = fmaxf(pmax, xb[(hh ^ 1) * 128 + row]) * a.sl2e;
        // rescale O only when the row max grew by more than 2^8 (both halves
        // decide alike: same inputs)
        const float m_new = (j == 0 || tmax > m + kRescaleLog2) ? tmax : m;
        const bool grow = j > 0 && m_new != m;
        if (__any_sync(0xffffffffu, grow)) {
          // O may be touched only once PV(g-1) is done.  PV(g-1) completes a
          // phase of o_done[(g-1)%2] that is at most one behind (S(g) is done,
          // so PV(g-3) is) and never ahead (PV(g+1) needs P(g+1)).
          ok = mbar_wait_warp(&o_done[2 * i + ((g - 1) & 1)], ((g - 1) >> 1) & 1);
          if (!ok) break;
          tc_fence_after_sync();
          const float alpha = grow ? ex2f(m - m_new) : 1.0f;
          float o[16];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            tmem_ld16(tO(i) + lane_off + 64 * hh + c * 16, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] *= alpha;
            tmem_st16(tO(i) + lane_off + 64 * hh + c * 16, o);
          }
          tmem_wait_st();
          l *= alpha;
        }
        m = m_new;
        // P = 2^(S*c - m) (masked entries -inf, so 0) as f16 pairs into TMEM
        // columns 16*hh .. 16*hh+15 of this S buffer
        const float2 c2 = make_float2(a.sl2e, a.sl2e), nm2 = make_float2(-m, -m);
        float2 ls = make_float2(0.f, 0.f);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 xv = ffma2(make_float2(v[e], v[e + 1]), c2, nm2);
          const float2 pe = make_float2(ex2f(xv.x), ex2f(xv.y));
          ls = make_float2(ls.x + pe.x, ls.y + pe.y);
          const __half2 hp = __floats2half2_rn(pe.x, pe.y);
          pk[e / 2] = *reinterpret_cast<const uint32_t*>(&hp);
        }
        l += ls.x + ls.y;
        // P(g) goes over S buffer g % 2, which PV(g-1) does not read; each
        // warp publishes its rows once its stores are done
        tmem_st16u(tS(i, g & 1) + lane_off + 16 * hh, pk);
        tmem_wait_st();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[2 * i + (g & 1)]);
      }
      if (!ok) break;
      // ---- the item's O: row sum of both halves, then O from TMEM once its
      // last PV is done; O is released to the next item as soon as it is read
      float* xs = xsum + i * 256;
      xs[hh * 128 + row] = l;
      ok = exchange();
      if (!ok) break;
      const float inv = 1.0f / (l + xs[(hh ^ 1) * 128 + row]);
      const int gl = g - 1;  // PV(gl) is the last; S(gl) is done, so PV(gl-2) is
      ok = mbar_wait_warp(&o_done[2 * i + (gl & 1)], (gl >> 1) & 1);
      if (!ok) break;
      tc_fence_after_sync();
      float* dst = a.out + (((int64_t)x.b * a.T + qidx) * a.Hq + x.h) * kPrefillHD + 64 * hh;
      const bool in_range = qidx < a.T;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        tmem_ld32(tO(i) + lane_off + 64 * hh + c * 32, v);
        tmem_wait_ld();
        if (c == 1) {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&o_free[i]);
        }
        if (in_range) {
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(dst + c * 32 + e) =
                make_float4(v[e] * inv, v[e + 1] * inv, v[e + 2] * inv, v[e + 3] * inv);
        }
      }
    }
    if (!ok && lane == 0) set_dev_err(a.dev_err, ASR_DEVERR_TIMEOUT);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 16) {
    tc_fence_after_sync();
    tmem_dealloc(tbase, 512);
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

// Checks shared by the prefill entry points (host only, before any launch).
static int prefill_check(int B, int T, int q_heads, int kv_heads, int head_dim, int capacity,
                         const void* cache, int64_t seq_stride, void* ws, size_t ws_bytes) {
  if (B < 0 || B > ASR_MAX_BATCH || T < 1 || q_heads < 1 || kv_heads < 1 || capacity < 1)
    return ASR_ERR_INVALID_ARG;
  if (head_dim != kPrefillHD || q_heads % kv_heads != 0 || kv_heads > 16 || q_heads > 64)
    return ASR_ERR_UNSUPPORTED;
  if (T > capacity) return ASR_ERR_INVALID_ARG;
  if (B == 0) return ASR_OK;
  if (!cache) return ASR_ERR_INVALID_ARG;
  if (seq_stride < (int64_t)capacity * 2 * kv_heads * head_dim) return ASR_ERR_INVALID_ARG;
  if (!aligned16(cache) || seq_stride % 8 != 0) return ASR_ERR_MISALIGNED;
  if (!ws || ((uintptr_t)ws & 255u) != 0 || ws_bytes < prefill_ws_bytes(B, T, q_heads, kv_heads))
    return ASR_ERR_WORKSPACE;
  return ASR_OK;
}

static cudaError_t prefill_attrs() {
  static cudaError_t attr = cudaSuccess;
  std::call_once(g_prefill_attr, [] {
    attr = cudaFuncSetAttribute(prefill_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kAttnSmem);
    if (attr == cudaSuccess)
      attr = cudaFuncSetAttribute(prefill_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  100 * 1024);
  });
  return attr;
}

static uint16_t* ws_vt(void* ws, int B, int T, int q_heads) {
  return reinterpret_cast<uint16_t*>(static_cast<char*>(ws) +
                                     align_up((size_t)B * T * q_heads * kPrefillHD * 2, 1024));
}

extern "C" int asr_prefill_prep(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                const float* q_norm_w, const float* k_norm_w, float eps,
                                float rope_base, int B, int T, int q_heads, int kv_heads,
                                int head_dim, uint16_t* cache, int64_t seq_stride, int capacity,
                                void* ws, size_t ws_bytes, asr_stream_t stream) {
  if (!(eps >= 0.f) || !(rope_base > 0.f)) return ASR_ERR_INVALID_ARG;
  int st = prefill_check(B, T, q_heads, kv_heads, head_dim, capacity, cache, seq_stride, ws,
                         ws_bytes);
  if (st != ASR_OK || B == 0) return st;
  if (!q || !k || !v || !q_norm_w || !k_norm_w) return ASR_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return ASR_ERR_MISALIGNED;
  if (prefill_attrs() != cudaSuccess) return ASR_ERR_CUDA;
  const int Tpad = round_up(T, 128);
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
  pa.qhat = static_cast<uint16_t*>(ws);
  pa.vt = ws_vt(ws, B, T, q_heads);
  for (int i = 0; i < kPrefillHD / 2; ++i)
    pa.theta[i] = pow((double)rope_base, -2.0 * i / kPrefillHD);
  const size_t prep_smem =
      2 * kPrepT * (kPrefillHD / 2) * sizeof(float) + (size_t)kPrepT * kv_heads * kPrefillHD * 2;
  cudaError_t e = launch_pdl(prefill_prep_kernel, dim3(Tpad / kPrepT, B), dim3(256), prep_smem,
                             (cudaStream_t)stream, pa);
  return e == cudaSuccess ? ASR_OK : ASR_ERR_CUDA;
}

extern "C" int asr_prefill_attention(int B, int T, int q_heads, int kv_heads, int head_dim,
                                     float scale, const uint16_t* cache, int64_t seq_stride,
                                     int capacity, float* out, void* ws, size_t ws_bytes,
                                     int32_t* dev_err, asr_stream_t stream) {
  int st = prefill_check(B, T, q_heads, kv_heads, head_dim, capacity, cache, seq_stride, ws,
                         ws_bytes);
  if (st != ASR_OK || B == 0) return st;
  if (!out) return ASR_ERR_INVALID_ARG;
  if (!aligned16(out)) return ASR_ERR_MISALIGNED;
  if (prefill_attrs() != cudaSuccess) return ASR_ERR_CUDA;
  const int Tpad = round_up(T, 128);
  const int64_t row = 2LL * kv_heads * kPrefillHD;
  // tensor maps: q^ (dims: Hq*128, T, B), cache (row, capacity, B), V^T (Tpad, 128, B*Hkv)
  CUtensorMap tq, tk, tv;
  if (!make_tmap_f16_3d(&tq, ws, (uint64_t)q_heads * kPrefillHD, T, B,
                        (uint64_t)q_heads * kPrefillHD * 2, (uint64_t)T * q_heads * kPrefillHD * 2,
                        64, 128) ||
      !make_tmap_f16_3d(&tk, cache, (uint64_t)row, capacity, B, (uint64_t)row * 2,
                        (uint64_t)seq_stride * 2, 64, 64) ||
      !make_tmap_f16_3d(&tv, ws_vt(ws, B, T, q_heads), Tpad, kPrefillHD, (uint64_t)B * kv_heads,
                        (uint64_t)Tpad * 2, (uint64_t)Tpad * kPrefillHD * 2, 64, 128))
    return ASR_ERR_CUDA;
  PrefillAttnArgs aa = {};
  aa.B = B;
  aa.T = T;
  aa.Hq = q_heads;
  aa.Hkv = kv_heads;
  aa.n_qt = (T + 127) / 128;
  aa.n_pairs = (aa.n_qt + 1) / 2;
  aa.n_items = aa.n_pairs * B * q_heads;
  aa.sl2e = scale * kLog2eP;
  aa.out = out;
  aa.dev_err = dev_err;
  const int sms = device_sm_count();
  if (sms <= 0) return ASR_ERR_CUDA;
  const int ctas = aa.n_items < sms ? aa.n_items : sms;  // persistent: one per SM
  cudaError_t e = launch_pdl(prefill_attn_kernel, dim3(ctas),
                             dim3(kAttnThreads), (size_t)kAttnSmem, (cudaStream_t)stream, tq, tk,
                             tv, aa);
  return e == cudaSuccess ? ASR_OK : ASR_ERR_CUDA;
}

extern "C" int asr_prefill_attn(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                const float* q_norm_w, const float* k_norm_w, float eps,
                                float rope_base, int B, int T, int q_heads, int kv_heads,
                                int head_dim, float scale, uint16_t* cache, int64_t seq_stride,
                                int capacity, float* out, void* ws, size_t ws_bytes,
                                int32_t* dev_err, asr_stream_t stream) {
  // every check of both stages first, so that a rejected call enqueues nothing
  if (!(eps >= 0.f) || !(rope_base > 0.f)) return ASR_ERR_INVALID_ARG;
  int st = prefill_check(B, T, q_heads, kv_heads, head_dim, capacity, cache, seq_stride, ws,
                         ws_bytes);
  if (st != ASR_OK || B == 0) return st;
  if (!q || !k || !v || !q_norm_w || !k_norm_w || !out) return ASR_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return ASR_ERR_MISALIGNED;
  st = asr_prefill_prep(q, k, v, q_norm_w, k_norm_w, eps, rope_base, B, T, q_heads, kv_heads,
                        head_dim, cache, seq_stride, capacity, ws, ws_bytes, stream);
  if (st != ASR_OK) return st;
  return asr_prefill_attention(B, T, q_heads, kv_heads, head_dim, scale, cache, seq_stride,
                               capacity, out, ws, ws_bytes, dev_err, stream);
}
