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
//   k^ = f16(RoPE_t(RMSNorm(k) * w_k)) (to cache row t), and V is copied to
//   cache row t.
// a8 attention (5th-generation tensor cores): one CTA per (pair of adjacent
//   128-query tiles, sequence, query head), warp-specialised.  Q, K and V tiles
//   arrive by tiled TMA with the 128-byte swizzle (V as the cache holds it,
//   read by the PV product as an MN-major operand; with per-sequence lengths
//   the MHA path reads a transposed, zero-padded V^T instead, K-major, so that
//   no key past a sequence's length reaches the product); S = Q K^T (128 x 64 per
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
  float rope_turns[kPrefillHD];  // theta_i / (2 pi) as float pairs (hi, lo), i < 64
};

// grid (Tpad / kPrepT, B), 256 threads.  Shared: cos/sin of the chunk's
// positions.
__global__ void __launch_bounds__(256) prefill_prep_kernel(const __grid_constant__ PrepArgs a) {
  constexpr int HD = kPrefillHD, HALF = HD / 2;
  extern __shared__ __align__(16) unsigned char psm[];
  float* cs = reinterpret_cast<float*>(psm);   // [kPrepT][HALF]
  float* sn = cs + kPrepT * HALF;              // [kPrepT][HALF]
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

  // rotation table: the angle t * theta_i in turns, theta_i / (2 pi) held as
  // an unevaluated float pair (hi + lo).  t * hi is split exactly into its
  // rounded value and error (fmaf); the whole turns are removed from the
  // rounded part exactly and the small terms added back, so the fraction f
  // carries about 2^-24 absolute error for any t < 2^24, and sincospif
  // evaluates sin/cos(pi * 2f) with its own trivial reduction.
  for (int idx = tid; idx < kPrepT * HALF; idx += blockDim.x) {
    const int tt = idx / HALF, i = idx % HALF;
    const float pf = (float)(t0 + tt);
    const float hi = a.rope_turns[2 * i], lo = a.rope_turns[2 * i + 1];
    const float prod = pf * hi;
    const float err = fmaf(pf, hi, -prod);
    const float f = (prod - rintf(prod)) + fmaf(pf, lo, err);
    float s, c;
    sincospif(2.0f * f, &s, &c);
    cs[idx] = c;
    sn[idx] = s;
  }
  // V rows: to the cache
#pragma unroll
  for (int u = 0; u < kPrepV; ++u) {
    const int idx = tid + u * (int)blockDim.x;
    if (idx < nv) {
      const int tt = idx / vec_per_row, c = idx % vec_per_row;
      if (t0 + tt < a.T)
        *reinterpret_cast<uint4*>(a.cache + (int64_t)b * a.seq_stride + (int64_t)(t0 + tt) * 2 * kw +
                                  kw + c * 8) = vval[u];
    }
  }
  // the rows past the first blockDim * kPrepV vectors (more KV heads than
  // the registers cover) go the plain way
  for (int idx = tid + kPrepV * (int)blockDim.x; idx < nv; idx += blockDim.x) {
    const int tt = idx / vec_per_row, c = idx % vec_per_row;
    if (t0 + tt < a.T) {
      const uint4 val = *reinterpret_cast<const uint4*>(a.v + ((int64_t)b * a.T + t0 + tt) * kw + c * 8);
      *reinterpret_cast<uint4*>(a.cache + (int64_t)b * a.seq_stride + (int64_t)(t0 + tt) * 2 * kw +
                                kw + c * 8) = val;
    }
  }
  __syncthreads();

  // normed + roped heads: half-warp hw owns position t0 + hw (256 threads =
  // 16 half-warps = kPrepT positions) and walks all its q and k heads, so
  // its cos/sin stay in registers and no index is divided.  Lane hl of the
  // half-warp holds dims 8*hl .. 8*hl+7, so lanes hl and hl ^ 8 hold NeoX
  // RoPE partners (i, i + 64).  kPrepU head vectors are loaded before any is
  // reduced, so several 16-byte loads per lane are in flight.
  constexpr int kPrepU = 4;
  const int hw = tid >> 4, hl = tid & 15;
  const bool upper = hl >= 8;
  const int ib = (hl & 7) * 8;  // frequency index of this lane's first dim
  float wqr[8], wkr[8], cr[8], sr[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    wqr[e] = a.wq[8 * hl + e];
    wkr[e] = a.wk[8 * hl + e];
    cr[e] = cs[hw * HALF + ib + e];
    sr[e] = sn[hw * HALF + ib + e];
  }
  const int t = t0 + hw;
  const bool live = t < a.T;
  const int nheads = a.Hq + a.Hkv;
  const uint16_t* qrow = a.q + ((int64_t)b * a.T + t) * a.Hq * HD;
  const uint16_t* krow = a.k + ((int64_t)b * a.T + t) * kw;
  uint16_t* qdst = a.qhat + ((int64_t)b * a.T + t) * a.Hq * HD;
  uint16_t* kdst = a.cache + (int64_t)b * a.seq_stride + (int64_t)t * 2 * kw;
  for (int base = 0; base < nheads; base += kPrepU) {
    uint4 x[kPrepU];
#pragma unroll
    for (int u = 0; u < kPrepU; ++u) {
      const int hh = base + u;
      x[u] = make_uint4(0u, 0u, 0u, 0u);
      if (live && hh < nheads)
        x[u] = *reinterpret_cast<const uint4*>(
            (hh < a.Hq ? qrow + hh * HD : krow + (hh - a.Hq) * HD) + 8 * hl);
    }
#pragma unroll
    for (int u = 0; u < kPrepU; ++u) {
      // every lane runs the shuffles (both half-warps of a warp walk the same heads)
      const int hh = base + u;
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
        y[e] = upper ? xn[e] * cr[e] + pe * sr[e] : xn[e] * cr[e] - pe * sr[e];
      }
      if (live && hh < nheads) {
        uint16_t* dst = is_q ? qdst + hh * HD : kdst + (hh - a.Hq) * HD;
        *reinterpret_cast<uint4*>(dst + 8 * hl) = f8_to_h8(y);
      }
    }
  }
}

// --------------------------------------------------------- MHA prep --

struct MhaPrepArgs {
  const uint16_t* k;  // [B][T][H*HD]
  const uint16_t* v;
  const int32_t* lens;  // or null
  int B, T, Tpad, H, HD;
  uint16_t* cache;  // or null: rows of [K(H*HD) | V(H*HD)], sequence stride seq_stride
  int64_t seq_stride;
  uint16_t* vt;  // [B*H][HD][Tpad]
  int write_vt;  // with per-sequence lengths: V^T, zero at and past each length
};

constexpr int kMhaPrepT = 64;  // positions per CTA

// grid (Tpad / 64, H, B), 256 threads: one head of 64 positions of one
// sequence per CTA.  Its V (and K) vectors are loaded and copied to the
// cache rows of the real positions; with per-sequence lengths V is also
// staged in shared memory, then written transposed (64 positions = 128 bytes
// per dim row), zero at and past the sequence's length.
__global__ void __launch_bounds__(256) mha_prep_kernel(const __grid_constant__ MhaPrepArgs a) {
  __shared__ __align__(16) uint16_t tile[kMhaPrepT][128 + 8];
  const int tid = threadIdx.x;
  const int h = blockIdx.y, b = blockIdx.z;
  const int t0 = blockIdx.x * kMhaPrepT;
  grid_launch_dependents();
  grid_dependency_wait();
  int L = a.T;
  if (a.lens) {
    L = a.lens[b];
    if (L < 0 || L > a.T) L = 0;
  }
  // the attention reads V^T up to the end of the sequence's last 128-key
  // tile (zero past the length) and never beyond it
  if (t0 >= (L + 127) / 128 * 128) return;
  const int HD = a.HD, vpr = HD / 8;  // 16-byte vectors per head row
  const int64_t rw = (int64_t)a.H * HD;
  for (int idx = tid; idx < kMhaPrepT * vpr; idx += blockDim.x) {
    const int tt = idx / vpr, c = idx % vpr, t = t0 + tt;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (t < L) {
      const int64_t off = ((int64_t)b * a.T + t) * rw + h * HD + c * 8;
      val = *reinterpret_cast<const uint4*>(a.v + off);
      if (a.cache) {
        const uint4 kv = *reinterpret_cast<const uint4*>(a.k + off);
        uint16_t* row = a.cache + (int64_t)b * a.seq_stride + (int64_t)t * 2 * rw;
        *reinterpret_cast<uint4*>(row + h * HD + c * 8) = kv;
        *reinterpret_cast<uint4*>(row + rw + h * HD + c * 8) = val;
      }
    }
    // 16-byte chunk c of position tt goes to chunk c ^ (tt / 8): the
    // column reads below then hit 32 different banks
    if (a.write_vt) *reinterpret_cast<uint4*>(&tile[tt][(c ^ ((tt >> 3) & 7)) * 8]) = val;
  }
  if (!a.write_vt) return;
  __syncthreads();
  for (int idx = tid; idx < HD * (kMhaPrepT / 8); idx += blockDim.x) {
    const int d = idx / (kMhaPrepT / 8), q8 = idx % (kMhaPrepT / 8);
    alignas(16) uint16_t col[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) col[e] = tile[q8 * 8 + e][(((d >> 3) ^ q8) << 3) + (d & 7)];
    *reinterpret_cast<uint4*>(a.vt + (((int64_t)b * a.H + h) * HD + d) * a.Tpad + t0 + q8 * 8) =
        *reinterpret_cast<const uint4*>(col);
  }
}

// ------------------------------------------------------------- attention --

struct PrefillAttnArgs {
  int B, T, Hq, Hkv, n_qt, n_pairs, n_items;
  int vcol0;    // without lengths: column of V head 0 in the rows tv maps
  float sl2e;   // scale * log2(e)
  float* out;   // [B][T][Hq*HD] fp32
  const int32_t* lens;  // real positions per sequence (device, [B]), or null: T for all
  int32_t* dev_err;
};

constexpr int kQBufs = 2;                 // Q tiles: one per slot (use n = 2*item + slot -> n % kQBufs)
constexpr int kStgBytes = 8 * 32 * 32 * 4;  // output staging: 32 rows x 32 fp32 per softmax warp
constexpr int kBarBytes = 1024;           // mbarriers and the TMEM address
constexpr int kAttnThreads = 320;  // warps 0-3, 4-7: softmax of slots A, B; 8: TMA; 9: MMA

// Tile sizes for head dimension HD (64 or 128).  Q, K and V tiles are 128
// rows (queries or keys) of HD dims, stored as HD/64 blocks of 128 rows x
// 128 bytes (the 128-byte swizzle atom); V^T tiles (with per-sequence
// lengths) are HD rows (dims) of 128 keys, as two 64-key blocks.  With head
// pairs (HP) a K or V^T stage holds the tiles of two heads.  The K/V ring is
// deeper when the tiles are smaller.
template <int HD, bool HP = false>
struct AttnCfg {
  static constexpr int QT = 128 * HD * 2, KT = (HP ? 2 : 1) * 128 * HD * 2;
  static constexpr int VT = (HP ? 2 : 1) * HD * 128 * 2;
  static constexpr int STAGES = (HD == 128 || HP) ? 2 : 4;
  static constexpr int SMEM = kQBufs * QT + STAGES * (KT + VT) + kStgBytes + kBarBytes + 1024;
};

// Head-pair items: the short-prompt multi-head prefill (head dim 64, causal,
// per-sequence lengths).
template <int HD, bool CAUSAL, bool VARLEN>
constexpr bool attn_head_pairs() {
  return HD == 64 && CAUSAL && VARLEN;
}
constexpr float kRescaleLog2 = 8.0f;      // rescale O only when the row max grows by > 2^8

// max of three fp32 values in one instruction (sm_100+)
__device__ __forceinline__ float fmax3(float x, float y, float z) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(x), "f"(y), "f"(z));
  return r;
}

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One work item: two query tiles of one sequence, tile qt_a of head h in
// slot A and tile qt_b of head hb in slot B.  Usually the two adjacent tiles
// 2p and 2p+1 of one head (h = hb), which share every K/V tile.  Head pairs
// (HP) put the same tile t of heads 2p and 2p+1 in the two slots instead
// (their K and V tiles are loaded together), so that short prompts, whose
// one or three tiles per head leave an adjacent pair half empty, keep both
// slots busy.  Key tiles are 128 keys.  Causal: a query tile visits the key
// tiles up to its own; unmasked: all key tiles of the sequence.  A tile at or
// past the sequence's real length L (lens[b]), or of a head past the last, is
// absent (0 tiles); an item with neither tile is empty.
struct PfItem {
  int b, h, hb, kvh, qt_a, qt_b, nA, nB, n, L;
};

// Head pairs list only the tiles that exist: tab holds the sequences ordered
// by their tile count, most first (tab[0 .. B)), then for each tile t the
// number of sequences that have it (tab[B + t]).  Item it runs tile t of
// the first tab[B + t] sequences, t from the last down, head pairs fastest.
template <bool CAUSAL, bool VARLEN, bool HP>
__device__ __forceinline__ PfItem pf_item(const PrefillAttnArgs& a, int it, const int* tab) {
  PfItem x;
  if constexpr (HP) {
    // items run longest tiles first
    const int hpairs = (a.Hq + 1) / 2;
    int t = a.n_qt - 1;
    while (t > 0 && it >= tab[a.B + t] * hpairs) {
      it -= tab[a.B + t] * hpairs;
      --t;
    }
    x.b = tab[it / hpairs];
    x.h = 2 * (it % hpairs);
    x.hb = x.h + 1;
    x.kvh = x.h;  // head pairs only without grouped queries
    x.qt_a = x.qt_b = t;
  } else {
    const int BH = a.B * a.Hq;
    const int pair = a.n_pairs - 1 - it / BH;  // items run longest pairs first
    const int bh = it % BH;
    x.b = bh / a.Hq;
    x.h = x.hb = bh % a.Hq;
    x.kvh = x.h / (a.Hq / a.Hkv);
    x.qt_a = 2 * pair;
    x.qt_b = 2 * pair + 1;
  }
  int L = a.T;
  if (VARLEN) {
    L = __ldg(a.lens + x.b);
    if (L < 0 || L > a.T) L = 0;  // reported by the producer warp
  }
  x.L = L;
  const int nt = (L + 127) / 128;  // query (and key) tiles of the sequence
  const bool b_ok = x.hb < a.Hq;
  if (CAUSAL) {
    x.nA = x.qt_a < nt ? x.qt_a + 1 : 0;
    x.nB = b_ok && x.qt_b < nt ? x.qt_b + 1 : 0;
  } else {
    x.nA = x.qt_a < nt ? nt : 0;
    x.nB = b_ok && x.qt_b < nt ? nt : 0;
  }
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
// roles.  Warps 0-3 and 4-7 run the softmax of slots A and B, one thread per
// query row (warp w reads TMEM lanes 32*(w%4)..+31) holding the row's 128
// scores of a key tile.  Warp 8 owns the TMEM allocation and issues the TMA
// loads (Q per item; K and V^T per 128-key tile through two-stage rings
// that run on across items).  Warp 9 issues the MMAs.  Each slot has one S
// buffer: while one slot's softmax turns its S into P, the tensor core runs
// the other slot's PV and next S (ping-pong), so with the softmax shorter
// than a slot's MMA work the tensor core stays busy.  K and V^T have rings
// of their own: K of a tile is free after its S products, one tile before
// its V^T, so the next K loads well ahead of its S.  Every barrier's phase
// is counted across items, so the next item's loads and first S products
// overlap the end of the current item.
template <int HD, bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(kAttnThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, const PrefillAttnArgs a) {
  constexpr bool HP = attn_head_pairs<HD, CAUSAL, VARLEN>();
  using C = AttnCfg<HD, HP>;
  constexpr int kQTile = C::QT, kKTile = C::KT, kVTile = C::VT, kKVStages = C::STAGES;
  constexpr int kHalfBlock = 128 * 128;  // bytes of one 64-dim block of a Q or K tile
  constexpr int kVHead = HD * 128 * 2;   // bytes of one head's V^T tile
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  unsigned char* sQ = smem;                                  // kQBufs Q tiles
  unsigned char* sK = sQ + kQBufs * kQTile;                  // stages x K tile
  unsigned char* sV = sK + kKVStages * kKTile;               // stages x V^T tile
  float* sStg = reinterpret_cast<float*>(sV + kKVStages * kVTile);  // 8 x 4 KB
  uint64_t* bar = reinterpret_cast<uint64_t*>(sV + kKVStages * kVTile + kStgBytes);
  uint64_t* q_full = bar;                   // kQBufs: the Q tile of a use landed
  uint64_t* q_empty = q_full + kQBufs;      // kQBufs: that use's S products are done with it
  uint64_t* k_full = q_empty + kQBufs;      // kKVStages each
  uint64_t* k_empty = k_full + kKVStages;
  uint64_t* v_full = k_empty + kKVStages;
  uint64_t* v_empty = v_full + kKVStages;
  uint64_t* s_full = v_empty + kKVStages;   // [A, B]: S of the slot's tile g (phase g)
  uint64_t* p_full = s_full + 2;            // [A0, A1, B0, B1]: half h (keys 64h..) of P of tile g
  uint64_t* o_done = p_full + 4;            // [A, B]: the slot's last PV of an item
  uint64_t* o_free = o_done + 2;            // [A, B]: the softmax has read O of its item
  uint64_t* drain = o_free + 2;             // every MMA this CTA issued has completed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_any = reinterpret_cast<int*>(tslot + 1);  // some wait of this CTA gave up
  // head pairs: the item table (see pf_item), after the barrier block
  int* tab = reinterpret_cast<int*>(reinterpret_cast<unsigned char*>(bar) + kBarBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int u = 0; u < kQBufs; ++u) {
      mbar_init(&q_full[u], 1);
      mbar_init(&q_empty[u], 1);
    }
    for (int s = 0; s < kKVStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_full[2 * i], 4);  // one arrival per softmax warp of the slot
      mbar_init(&p_full[2 * i + 1], 4);
      mbar_init(&o_done[i], 1);
      mbar_init(&o_free[i], 4);
    }
    mbar_init(drain, 1);
    *abort_any = 0;
    fence_barrier_init();
  }
  if (warp == 8) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  grid_launch_dependents();
  grid_dependency_wait();
  if constexpr (HP) {
    if (warp == 0) {
      // sequences by tile count, most first (one ballot per 32 sequences
      // and count), and per tile the number of sequences that have it; the
      // item count last.  A bad length is reported here (its sequence has
      // no tiles, so no item would).
      int pos = 0;
      for (int v = a.n_qt; v >= 1; --v) {
        for (int b0 = 0; b0 < a.B; b0 += 32) {
          const int b = b0 + lane;
          int L = 0;
          if (b < a.B) {
            L = __ldg(a.lens + b);
            if (L < 0 || L > a.T) {
              if (v == a.n_qt && blockIdx.x == 0) set_dev_err(a.dev_err, ASR_DEVERR_LEN);
              L = 0;
            }
          }
          const bool hit = b < a.B && (L + 127) / 128 == v;
          const unsigned m = __ballot_sync(0xffffffffu, hit);
          if (hit) tab[pos + __popc(m & ((1u << lane) - 1u))] = b;
          pos += __popc(m);
        }
        if (lane == 0) tab[a.B + v - 1] = pos;
      }
      __syncwarp();
      if (lane == 0) {
        int items = 0;
        for (int t = 0; t < a.n_qt; ++t) items += tab[a.B + t];
        tab[a.B + a.n_qt] = items * ((a.Hq + 1) / 2);
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = *tslot;
  // items of this launch: head pairs count only the tiles that exist
  const int n_items = HP ? tab[a.B + a.n_qt] : a.n_items;
  // TMEM columns: S/P of slot i at 128*i (P: 128 keys packed two per column
  // over the first 64), O_A at 256, O_B at 384.
  auto tS = [&](int i) { return tbase + 128u * i; };
  auto tO = [&](int i) { return tbase + 256u + 128u * i; };

  int nk = 0, nv = 0, nq = 0;  // producer: K, V tile copies and Q uses issued
  if (warp == 8) {
    // ======================================================= TMA producer
    // The whole warp runs the schedule; one elected lane issues each copy.
    // Q tiles rotate through kQBufs buffers: use n = 2*item + slot takes
    // buffer n % kQBufs, so the next item's slot-A tile lands in the buffer
    // the previous item's slot B has finished with, while this item runs.
    int gk = 0;  // K/V tiles loaded so far (ring position)
    bool ok = true;
    // Q tile of slot i of item k (x): wait until the buffer's previous use
    // is done, then load (a slot with no tile completes its phase with no
    // bytes)
    auto load_q = [&](int k, int i, const PfItem& x) {
      const int n = 2 * k + i, u = n % kQBufs, c = n / kQBufs;
      if (c > 0 && !(ok = mbar_wait_warp(&q_empty[u], (c - 1) & 1))) return;
      const bool has = (i == 0 ? x.nA : x.nB) > 0;
      mbar_arrive_expect_tx_warp(&q_full[u], has ? kQTile : 0);
      ++nq;
      if (has) {
        const int qt = i == 0 ? x.qt_a : x.qt_b, qh = i == 0 ? x.h : x.hb;
        unsigned char* qd = sQ + u * kQTile;
#pragma unroll
        for (int c = 0; c < HD / 64; ++c)
          tma_load_3d_warp(qd + c * kHalfBlock, &tq, qh * HD + 64 * c, qt * 128, x.b, &q_full[u]);
      }
    };
    for (int k = 0; ok; ++k) {
      const int it = pf_item_index(k, n_items);
      if (it < 0) break;
      const PfItem x = pf_item<CAUSAL, VARLEN, HP>(a, it, tab);
      if (VARLEN && x.h == 0 && x.qt_a == 0 && lane == 0) {
        const int v = __ldg(a.lens + x.b);
        if (v < 0 || v > a.T) set_dev_err(a.dev_err, ASR_DEVERR_LEN);
      }
      load_q(k, 0, x);  // its buffer was freed during the previous item
      for (int j = 0; j < x.n && ok; ++j, ++gk) {
        const int s = gk % kKVStages;
        const uint32_t ph = ((gk / kKVStages) - 1) & 1;
        unsigned char* kd = sK + s * kKTile;
        unsigned char* vd = sV + s * kVTile;
        if (gk >= kKVStages && !(ok = mbar_wait_warp(&k_empty[s], ph))) break;
        mbar_arrive_expect_tx_warp(&k_full[s], kKTile);
        ++nk;
        // (head pairs: heads kvh and kvh + 1, whose columns are adjacent)
#pragma unroll
        for (int c = 0; c < kKTile / kHalfBlock; ++c)
          tma_load_3d_warp(kd + c * kHalfBlock, &tk, x.kvh * HD + 64 * c, j * 128, x.b, &k_full[s]);
        if (gk >= kKVStages && !(ok = mbar_wait_warp(&v_empty[s], ph))) break;
        mbar_arrive_expect_tx_warp(&v_full[s], kVTile);
        ++nv;
        if constexpr (VARLEN) {
          // V^T rows (dims) of 128 keys, as two 64-key blocks (head pairs:
          // of each head)
#pragma unroll
          for (int hh = 0; hh < kVTile / kVHead; ++hh) {
            const int z = x.b * a.Hkv + x.kvh + hh;
            tma_load_3d_warp(vd + hh * kVHead, &tv, j * 128, 0, z, &v_full[s]);
            tma_load_3d_warp(vd + hh * kVHead + kVHead / 2, &tv, j * 128 + 64, 0, z, &v_full[s]);
          }
        } else {
          // V rows as they lie (keys x HD dims, HD/64 blocks of 128 keys x
          // 128 bytes): the PV product reads them MN-major
#pragma unroll
          for (int c = 0; c < HD / 64; ++c)
            tma_load_3d_warp(vd + c * kHalfBlock, &tv, a.vcol0 + x.kvh * HD + 64 * c, j * 128, x.b,
                             &v_full[s]);
        }
        if (j == 0) load_q(k, 1, x);  // the buffer of this item's slot A tile's predecessor
      }
      if (VARLEN && ok && x.n == 0) load_q(k, 1, x);  // an empty item still completes its slot B use
    }
    if (!ok && lane == 0) {
      set_dev_err(a.dev_err, ASR_DEVERR_TIMEOUT);
      atomicExch(abort_any, 1);
    }
  } else if (warp == 9) {
    // ======================================================= MMA issuer
    // The whole warp runs the schedule (operand descriptors stay
    // warp-uniform); one elected lane issues each tcgen05 operation.
    constexpr uint32_t kIdS = mma_idesc_f16_f32(128, 128);   // S = Q K^T: 128 x 128
    constexpr uint32_t kIdO = mma_idesc_f16_f32(128, HD);    // O += P V: 128 x HD
    constexpr uint32_t kIdOmn = mma_idesc_f16_f32_bmn(128, HD);  // ... with V rows as B
    const uint32_t aQ = smem_addr(sQ), aK = smem_addr(sK), aV = smem_addr(sV);
    int gk = 0;          // K/V tiles consumed so far
    int gx[2] = {0, 0};  // tiles of slot A / B so far (S and P phases)
    int ox[2] = {0, 0};  // items whose O slot A / B has accumulated so far
    bool ok = true;
    bool a_early = false;  // slot A's first S of this item was issued during the previous one
    for (int k = 0; ok; ++k) {
      const int it = pf_item_index(k, n_items);
      if (it < 0) break;
      const PfItem x = pf_item<CAUSAL, VARLEN, HP>(a, it, tab);
      const int nX[2] = {x.nA, x.nB};
      // Q buffer of slot i (use 2k + i) and the wait for its tile
      const int qb[2] = {(2 * k) % kQBufs, (2 * k + 1) % kQBufs};
      auto q_ready = [&](int i) {
        const int n = 2 * k + i;
        return mbar_wait_warp(&q_full[n % kQBufs], (n / kQBufs) & 1);
      };
      // S of slot i from Q buffer qbuf and K stage st; the slot's S buffer
      // holds P of its previous tile, read by a PV issued before this S
      auto issue_s_at = [&](int i, int qbuf, int st, bool last) {
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalfBlock + (kk & 3) * 32;
          const uint32_t koff = (kk >> 2) * kHalfBlock + (kk & 3) * 32;
          mma_f16_warp(tS(i), sw128_kmajor_desc(aQ + qbuf * kQTile + off),
                       sw128_kmajor_desc(aK + st * kKTile + (HP ? i * kHalfBlock : 0) + koff),
                       kIdS, kk > 0);
        }
        mma_commit_warp(&s_full[i]);
        if (last) mma_commit_warp(&q_empty[qbuf]);  // its Q free once these finish
      };
      auto issue_s = [&](int i, int j) {
        issue_s_at(i, qb[i], (gk + j) % kKVStages, j == nX[i] - 1);
      };
      // O += P V for keys 64h .. 64h+63 of key tile j: P (TMEM, 8 columns
      // per 16 keys) times the 64-key half h of V^T (shared memory)
      auto issue_pv_half = [&](int i, int j, int h) {
        const int st = (gk + j) % kKVStages;
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int kk = 4 * h + k4;
          if constexpr (VARLEN)
            mma_f16_ts_warp(tO(i), tS(i) + kk * 8,
                            sw128_kmajor_desc(aV + st * kVTile + (HP ? i * kVHead : 0) +
                                              h * (kVHead / 2) + k4 * 32),
                            kIdO, (j > 0 || kk > 0) ? 1u : 0u);
          else  // keys 16kk .. 16kk+15 are rows 16kk.. of each 64-dim block
            mma_f16_ts_warp(tO(i), tS(i) + kk * 8,
                            sw128_mnmajor_desc(aV + st * kVTile + kk * 2048, kHalfBlock), kIdOmn,
                            (j > 0 || kk > 0) ? 1u : 0u);
        }
        if (h == 1 && j == nX[i] - 1) mma_commit_warp(&o_done[i]);  // the item's O is complete
      };
      // K of tile j is free once both slots' S products for it are issued
      // (commit: once they finish); V^T of tile j once both slots' PVs are
      auto k_ready = [&](int j) {
        return mbar_wait_warp(&k_full[(gk + j) % kKVStages], ((gk + j) / kKVStages) & 1);
      };
      if (VARLEN && x.n == 0) {  // an empty item: release both Q uses and move on
        ok = q_ready(0) && q_ready(1);
        if (ok) {
          mma_commit_warp(&q_empty[qb[0]]);
          mma_commit_warp(&q_empty[qb[1]]);
        }
        continue;
      }
      ok = k_ready(0) && (a_early || q_ready(0));
      tc_fence_after_sync();
      if (ok && !a_early) issue_s(0, 0);
      a_early = false;
      if (ok) ok = q_ready(1);
      tc_fence_after_sync();
      if (ok && x.nB > 0) issue_s(1, 0);
      if (ok && x.nB == 0) mma_commit_warp(&q_empty[qb[1]]);  // slot B's unused buffer
      if (ok) mma_commit_warp(&k_empty[gk % kKVStages]);
      for (int j = 0; j < x.n && ok; ++j) {
        const int st = (gk + j) % kKVStages;
        ok = mbar_wait_warp(&v_full[st], ((gk + j) / kKVStages) & 1);
        if (ok && j + 1 < x.n) ok = k_ready(j + 1);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (ok && j < nX[i]) {
            const int g = gx[i] + j;
            // the first half of P goes to the tensor core while the softmax
            // still computes the second
            ok = mbar_wait_warp(&p_full[2 * i], g & 1);
            // the first PV of an item overwrites O: the softmax must have
            // read the previous item's O first
            if (ok && j == 0 && ox[i] > 0) ok = mbar_wait_warp(&o_free[i], (ox[i] - 1) & 1);
            tc_fence_after_sync();
            if (ok) issue_pv_half(i, j, 0);
            if (ok) ok = mbar_wait_warp(&p_full[2 * i + 1], g & 1);
            tc_fence_after_sync();
            if (ok) issue_pv_half(i, j, 1);
            if (ok && j + 1 < nX[i]) issue_s(i, j + 1);
          }
        }
        mma_commit_warp(&v_empty[st]);                               // V^T of tile j
        if (j + 1 < x.n) mma_commit_warp(&k_empty[(gk + j + 1) % kKVStages]);  // K of tile j+1
        // Slot A is done one tile before slot B: start its part of the next
        // item now (its Q is already in; its first K tile lands in the stage
        // this item's tile j has left), while slot B's softmax finishes.
        if (ok && j == x.nA - 1 && x.nB > x.nA) {
          const int it2 = pf_item_index(k + 1, n_items);
          if (it2 >= 0 && (!VARLEN || pf_item<CAUSAL, VARLEN, HP>(a, it2, tab).nA > 0)) {
            const PfItem x2 = pf_item<CAUSAL, VARLEN, HP>(a, it2, tab);
            const int g0 = gk + x.n, n2 = 2 * (k + 1);
            ok = mbar_wait_warp(&k_full[g0 % kKVStages], (g0 / kKVStages) & 1) &&
                 mbar_wait_warp(&q_full[n2 % kQBufs], (n2 / kQBufs) & 1);
            tc_fence_after_sync();
            if (ok) issue_s_at(0, n2 % kQBufs, g0 % kKVStages, x2.nA == 1);
            a_early = ok;
          }
        }
      }
      gx[0] += x.nA;
      gx[1] += x.nB;
      ox[0] += x.nA > 0 ? 1 : 0;
      ox[1] += x.nB > 0 ? 1 : 0;
      gk += x.n;
    }
    if (!ok && lane == 0) {
      set_dev_err(a.dev_err, ASR_DEVERR_TIMEOUT);
      atomicExch(abort_any, 1);
    }
  } else {
    // ======================================================= softmax
    const int i = warp >> 2;                  // 0: slot A, 1: slot B
    const int row = (warp & 3) * 32 + lane;   // 0..127: TMEM lane = query row
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    int g = 0;   // tiles of this slot so far (phase of s_full / p_full)
    int ox = 0;  // items of this slot so far (phase of o_done)
    bool ok = true;
    float v[128];
    for (int k = 0; ok; ++k) {
      const int it = pf_item_index(k, n_items);
      if (it < 0) break;
      const PfItem x = pf_item<CAUSAL, VARLEN, HP>(a, it, tab);
      const int ni = i == 0 ? x.nA : x.nB;
      if (ni == 0) continue;
      const int q0 = (i == 0 ? x.qt_a : x.qt_b) * 128;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < ni && ok; ++j, ++g) {
        // S(g) done also means the slot's PV(g-1) is done: it was issued
        // before S(g), and tcgen05 operations of one thread complete in order
        ok = mbar_wait_warp(&s_full[i], g & 1);
        if (!ok) break;
        tc_fence_after_sync();
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS(i) + lane_off + 32 * c, v + 32 * c);
        tmem_wait_ld();
        if (j == ni - 1) {
          // causal: the diagonal tile, keys past the row are masked (keys
          // past the length are past every real row); unmasked: the last
          // tile, keys at or past the length are masked
          const int lim = CAUSAL ? row : x.L - 1 - 128 * j;
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c > lim) v[c] = -INFINITY;
        }
        float mx[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          mx[e] = fmax3(fmax3(v[e], v[e + 16], v[e + 32]), fmax3(v[e + 48], v[e + 64], v[e + 80]),
                        fmaxf(v[e + 96], v[e + 112]));
#pragma unroll
        for (int e = 0; e < 5; ++e) mx[e] = fmax3(mx[3 * e], mx[3 * e + 1], mx[3 * e + 2]);
        const float tmax = fmax3(fmax3(mx[0], mx[1], mx[2]), fmaxf(mx[3], mx[4]), mx[15]) * a.sl2e;
        // rescale O only when the row max grew by more than 2^8
        const float m_new = (j == 0 || tmax > m + kRescaleLog2) ? tmax : m;
        const bool grow = j > 0 && m_new != m;
        if (__any_sync(0xffffffffu, grow)) {
          const float alpha = grow ? ex2f(m - m_new) : 1.0f;
          float o[16];
#pragma unroll 1
          for (int c = 0; c < HD / 16; ++c) {
            tmem_ld16(tO(i) + lane_off + c * 16, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) o[e] *= alpha;
            tmem_st16(tO(i) + lane_off + c * 16, o);
          }
          tmem_wait_st();
          l *= alpha;
        }
        m = m_new;
        // P = 2^(S*c - m) (masked entries -inf, so 0) as f16 pairs into the
        // first 64 columns of the S buffer (all of S is in registers)
        // P half h (keys 64h ..) is published as soon as it is stored, so
        // the tensor core starts on it while the other half is computed
        const float2 c2 = make_float2(a.sl2e, a.sl2e), nm2 = make_float2(-m, -m);
        float2 ls[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          ls[c] = make_float2(0.f, 0.f);
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 xv = ffma2(make_float2(v[32 * c + e], v[32 * c + e + 1]), c2, nm2);
            const float2 pe = make_float2(ex2f(xv.x), ex2f(xv.y));
            ls[c] = fadd2(ls[c], pe);
            const __half2 hp = __floats2half2_rn(pe.x, pe.y);
            pk[e / 2] = *reinterpret_cast<const uint32_t*>(&hp);
          }
          tmem_st16u(tS(i) + lane_off + 16 * c, pk);
          if (c & 1) {
            tmem_wait_st();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[2 * i + (c >> 1)]);
          }
        }
        l += (ls[0].x + ls[0].y) + (ls[1].x + ls[1].y) + ((ls[2].x + ls[2].y) + (ls[3].x + ls[3].y));
      }
      if (!ok) break;
      // ---- the item's O once its last PV is done; O is released to the
      // next item as soon as it is in registers
      ok = mbar_wait_warp(&o_done[i], ox & 1);
      ++ox;
      if (!ok) break;
      tc_fence_after_sync();
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) tmem_ld32(tO(i) + lane_off + 32 * c, v + 32 * c);
      tmem_wait_ld();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_free[i]);
      // The normalised rows go out through this warp's 4 KB of shared
      // memory, 32 columns at a time: each thread writes its row's 32
      // values, then each store instruction carries four whole 128-byte row
      // pieces instead of 32 rows' 16 bytes.  16-byte chunk c of row r sits
      // at chunk c ^ (r % 8), so both sides are free of bank conflicts.
      {
        const float inv = 1.0f / l;
        float* stg = sStg + warp * (32 * 32);
        const int r0 = q0 + (warp & 3) * 32;  // query row of lane 0
#pragma unroll
        for (int pc = 0; pc < HD / 32; ++pc) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int e = pc * 32 + c * 4;
            *reinterpret_cast<float4*>(stg + lane * 32 + ((c ^ (lane & 7)) * 4)) =
                make_float4(v[e] * inv, v[e + 1] * inv, v[e + 2] * inv, v[e + 3] * inv);
          }
          __syncwarp();
#pragma unroll
          for (int it = 0; it < 8; ++it) {
            const int rr = it * 4 + (lane >> 3), cc = lane & 7;
            const float4 val =
                *reinterpret_cast<const float4*>(stg + rr * 32 + ((cc ^ (rr & 7)) * 4));
            if (r0 + rr < x.L)
              *reinterpret_cast<float4*>(
                  a.out + (((int64_t)x.b * a.T + r0 + rr) * a.Hq + (i == 0 ? x.h : x.hb)) * HD +
                          pc * 32 + cc * 4) =
                  val;
          }
          __syncwarp();
        }
      }
    }
    if (!ok && lane == 0) {
      set_dev_err(a.dev_err, ASR_DEVERR_TIMEOUT);
      atomicExch(abort_any, 1);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  // After any wait of this CTA gave up, nothing may still be in flight into
  // its shared memory or tensor memory when it frees them and leaves: the
  // producer waits (bounded) for the copies it issued (only the last ring's
  // worth of K and V tiles and the last use of each Q buffer can be
  // pending), the MMA warp for every MMA it issued (a commit tracks all of
  // them).
  if (*reinterpret_cast<volatile int*>(abort_any)) {
    if (warp == 8) {
      for (int i = max(0, nk - kKVStages); i < nk; ++i)
        mbar_wait_warp(&k_full[i % kKVStages], (i / kKVStages) & 1);
      for (int i = max(0, nv - kKVStages); i < nv; ++i)
        mbar_wait_warp(&v_full[i % kKVStages], (i / kKVStages) & 1);
      for (int n = max(0, nq - kQBufs); n < nq; ++n)
        mbar_wait_warp(&q_full[n % kQBufs], (n / kQBufs) & 1);
    } else if (warp == 9) {
      mma_commit_warp(drain);
      mbar_wait_warp(drain, 0);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 8) {
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

bool make_tmap_f16_5d_plain(CUtensorMap* map, const void* base, const uint64_t dims[5],
                            const uint64_t strides_bytes[4], const uint32_t box[5]) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], estr[5];
  for (int i = 0; i < 5; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    estr[i] = 1;
  }
  for (int i = 0; i < 4; ++i) st[i] = strides_bytes[i];
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5, const_cast<void*>(base), d, st, bx, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static int round_up(int x, int m) { return (x + m - 1) / m * m; }

size_t prefill_ws_bytes(int B, int T, int Hq, int Hkv) {
  (void)Hkv;  // V is read from the cache rows
  return align_up((size_t)B * T * Hq * kPrefillHD * 2, 1024);
}

size_t mha_ws_bytes(int B, int T, int H, int HD) {
  return (size_t)B * H * HD * round_up(T, 128) * 2;  // V^T
}

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
  return ensure_dynamic_smem((const void*)prefill_prep_kernel, 100 * 1024);
}

// Launch the tensor-core attention for head dimension HD, causal or not.
// Q tiles are read through tq (dims: Hq*HD, T, B), K tiles through tk (a row
// buffer whose head h key vector sits at column h*HD), V^T through tv (dims:
// Tpad, HD, B*Hkv).  Persistent: one CTA per SM, at most one per item.
template <int HD, bool CAUSAL, bool VARLEN>
static int launch_attn_tc_v(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            PrefillAttnArgs& aa, cudaStream_t stream) {
  constexpr bool HP = attn_head_pairs<HD, CAUSAL, VARLEN>();
  if (HP && aa.Hq != aa.Hkv) return ASR_ERR_UNSUPPORTED;  // head pairs share no K/V head
  aa.n_qt = (aa.T + 127) / 128;
  // head pairs: the item table (sequences, tile counts, item count)
  const int smem =
      AttnCfg<HD, HP>::SMEM + (HP ? (int)align_up((size_t)(aa.B + aa.n_qt + 1) * 4, 16) : 0);
  if (smem > 227 * 1024) return ASR_ERR_UNSUPPORTED;
  if (ensure_dynamic_smem((const void*)attn_tc_kernel<HD, CAUSAL, VARLEN>, smem) != cudaSuccess)
    return ASR_ERR_CUDA;
  aa.n_pairs = (aa.n_qt + 1) / 2;
  aa.n_items = HP ? aa.n_qt * aa.B * ((aa.Hq + 1) / 2) : aa.n_pairs * aa.B * aa.Hq;
  const int sms = device_sm_count();
  if (sms <= 0) return ASR_ERR_CUDA;
  const int ctas = aa.n_items < sms ? aa.n_items : sms;
  cudaError_t e = launch_pdl(attn_tc_kernel<HD, CAUSAL, VARLEN>, dim3(ctas), dim3(kAttnThreads),
                             (size_t)smem, stream, tq, tk, tv, aa);
  return e == cudaSuccess ? ASR_OK : ASR_ERR_CUDA;
}

// With per-sequence lengths the kernel reads them per item and may meet
// empty items; without, that work is compiled out.
template <int HD, bool CAUSAL>
static int launch_attn_tc(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          PrefillAttnArgs& aa, cudaStream_t stream) {
  return aa.lens ? launch_attn_tc_v<HD, CAUSAL, true>(tq, tk, tv, aa, stream)
                 : launch_attn_tc_v<HD, CAUSAL, false>(tq, tk, tv, aa, stream);
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
  for (int i = 0; i < kPrefillHD / 2; ++i) {
    const double t = pow((double)rope_base, -2.0 * i / kPrefillHD) / (2.0 * 3.14159265358979323846);
    const float hi = (float)t;
    pa.rope_turns[2 * i] = hi;
    pa.rope_turns[2 * i + 1] = (float)(t - (double)hi);
  }
  const size_t prep_smem = 2 * kPrepT * (kPrefillHD / 2) * sizeof(float);
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
  const int64_t row = 2LL * kv_heads * kPrefillHD;
  // tensor maps: q^ (dims: Hq*128, T, B); the cache rows (row, capacity, B)
  // for K; the same rows cut at T (row, T, B) for V, so that the keys of the
  // last tile past T read as zero
  CUtensorMap tq, tk, tv;
  if (!make_tmap_f16_3d(&tq, ws, (uint64_t)q_heads * kPrefillHD, T, B,
                        (uint64_t)q_heads * kPrefillHD * 2, (uint64_t)T * q_heads * kPrefillHD * 2,
                        64, 128) ||
      !make_tmap_f16_3d(&tk, cache, (uint64_t)row, capacity, B, (uint64_t)row * 2,
                        (uint64_t)seq_stride * 2, 64, 128) ||
      !make_tmap_f16_3d(&tv, cache, (uint64_t)row, T, B, (uint64_t)row * 2,
                        (uint64_t)seq_stride * 2, 64, 128))
    return ASR_ERR_CUDA;
  PrefillAttnArgs aa = {};
  aa.vcol0 = kv_heads * kPrefillHD;  // V head 0 follows the K heads in a row
  aa.B = B;
  aa.T = T;
  aa.Hq = q_heads;
  aa.Hkv = kv_heads;
  aa.sl2e = scale * kLog2eP;
  aa.out = out;
  aa.lens = nullptr;
  aa.dev_err = dev_err;
  return launch_attn_tc<kPrefillHD, true>(tq, tk, tv, aa, (cudaStream_t)stream);
}

// Checks shared by the MHA entry points (host only, before any launch).
static int mha_check(const uint16_t* q, const uint16_t* k, const uint16_t* v, int B, int T,
                     int heads, int head_dim, const float* out, void* ws, size_t ws_bytes) {
  if (B < 0 || B > ASR_MAX_BATCH || T < 1 || heads < 1) return ASR_ERR_INVALID_ARG;
  if ((head_dim != 64 && head_dim != 128) || heads > ASR_MAX_KV_HEADS) return ASR_ERR_UNSUPPORTED;
  if (B == 0) return ASR_OK;
  if (!q || !k || !v || !out) return ASR_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return ASR_ERR_MISALIGNED;
  if (!ws || ((uintptr_t)ws & 255u) != 0 || ws_bytes < mha_ws_bytes(B, T, heads, head_dim))
    return ASR_ERR_WORKSPACE;
  return ASR_OK;
}

// The MHA prep (cache rows when cache is given; V^T with per-sequence
// lengths) then the tensor-core attention with Q and K read where they lie:
// K from the cache rows (prefill) or from k itself (encoder), and V from v
// itself (no lengths: the map is cut at T, so keys past T read as zero) or
// from V^T (lengths: keys past a sequence's length must read as zero, and
// rows of v past it may hold anything).
static int mha_run(const uint16_t* q, const uint16_t* k, const uint16_t* v, const int32_t* lens,
                   int B, int T, int heads, int head_dim, float scale, bool causal, uint16_t* cache,
                   int64_t seq_stride, float* out, void* ws, int32_t* dev_err,
                   cudaStream_t stream) {
  const int Tpad = round_up(T, 128);
  const bool use_vt = lens != nullptr;
  if (use_vt || cache) {
    MhaPrepArgs pa = {};
    pa.k = k;
    pa.v = v;
    pa.lens = lens;
    pa.B = B;
    pa.T = T;
    pa.Tpad = Tpad;
    pa.H = heads;
    pa.HD = head_dim;
    pa.cache = cache;
    pa.seq_stride = seq_stride;
    pa.vt = static_cast<uint16_t*>(ws);
    pa.write_vt = use_vt ? 1 : 0;
    if (launch_pdl(mha_prep_kernel, dim3(Tpad / kMhaPrepT, heads, B), dim3(256), 0, stream, pa) !=
        cudaSuccess)
      return ASR_ERR_CUDA;
  }
  const uint64_t rw = (uint64_t)heads * head_dim;
  CUtensorMap tq, tk, tv;
  bool ok = make_tmap_f16_3d(&tq, q, rw, T, B, rw * 2, (uint64_t)T * rw * 2, 64, 128);
  if (use_vt)
    ok = ok && make_tmap_f16_3d(&tv, ws, Tpad, head_dim, (uint64_t)B * heads, (uint64_t)Tpad * 2,
                                (uint64_t)Tpad * head_dim * 2, 64, head_dim);
  else
    ok = ok && make_tmap_f16_3d(&tv, v, rw, T, B, rw * 2, (uint64_t)T * rw * 2, 64, 128);
  if (cache)  // rows of [K | V] of 2*rw elements; K of head h at column h*hd
    ok = ok && make_tmap_f16_3d(&tk, cache, 2 * rw, T, B, 2 * rw * 2, (uint64_t)seq_stride * 2,
                                64, 128);
  else
    ok = ok && make_tmap_f16_3d(&tk, k, rw, T, B, rw * 2, (uint64_t)T * rw * 2, 64, 128);
  if (!ok) return ASR_ERR_CUDA;
  PrefillAttnArgs aa = {};
  aa.B = B;
  aa.T = T;
  aa.Hq = heads;
  aa.Hkv = heads;
  aa.vcol0 = 0;
  aa.sl2e = scale * kLog2eP;
  aa.out = out;
  aa.lens = lens;
  aa.dev_err = dev_err;
  if (head_dim == 64)
    return causal ? launch_attn_tc<64, true>(tq, tk, tv, aa, stream)
                  : launch_attn_tc<64, false>(tq, tk, tv, aa, stream);
  return causal ? launch_attn_tc<128, true>(tq, tk, tv, aa, stream)
                : launch_attn_tc<128, false>(tq, tk, tv, aa, stream);
}

extern "C" int asr_mha_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                               const int32_t* lens, int B, int T, int heads, int head_dim,
                               float scale, uint16_t* cache, int64_t seq_stride, int capacity,
                               float* out, void* ws, size_t ws_bytes, int32_t* dev_err,
                               asr_stream_t stream) {
  int st = mha_check(q, k, v, B, T, heads, head_dim, out, ws, ws_bytes);
  if (st != ASR_OK || B == 0) return st;
  if (capacity < 1 || T > capacity || !cache) return ASR_ERR_INVALID_ARG;
  if (seq_stride < (int64_t)capacity * 2 * heads * head_dim) return ASR_ERR_INVALID_ARG;
  if (!aligned16(cache) || seq_stride % 8 != 0) return ASR_ERR_MISALIGNED;
  return mha_run(q, k, v, lens, B, T, heads, head_dim, scale, true, cache, seq_stride, out, ws,
                 dev_err, (cudaStream_t)stream);
}

extern "C" int asr_encoder_attn(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                const int32_t* lens, int B, int T, int heads, int head_dim,
                                float scale, float* out, void* ws, size_t ws_bytes,
                                int32_t* dev_err, asr_stream_t stream) {
  int st = mha_check(q, k, v, B, T, heads, head_dim, out, ws, ws_bytes);
  if (st != ASR_OK || B == 0) return st;
  return mha_run(q, k, v, lens, B, T, heads, head_dim, scale, false, nullptr, 0, out, ws,
                 dev_err, (cudaStream_t)stream);
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
