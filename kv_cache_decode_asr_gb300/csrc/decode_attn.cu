// decode_attn.cu -- one-token attention over f16 K/V caches (a2, a3, a4, a5).
//
// Method: split-K flash-decoding with a log-sum-exp combine.  Every
// (source, key) pair of a call is laid on one flattened key axis (source =
// the sequence for self-attention and the GQA step, the beam group for
// cross-attention) and a persistent grid of P CTAs takes equal contiguous
// shares of it, so variable lengths stay balanced to within one tile.  A CTA
// streams its share as tiles of whole cache rows (K and V of every head are
// contiguous in a row) with one bulk TMA copy per tile into a multi-stage
// shared-memory ring (mbarrier full/empty pairs, one producer warp).  The
// consumer threads form groups of HD/8 lanes; a group owns one KV head and
// 8 dims per lane, keeps its queries (all beams of the group x all query
// heads of the KV head) in registers, and runs an online softmax in the log2
// domain over the rows it is given.  At the end of a source's piece the row
// slots are merged in shared memory; a source split over several CTAs leaves
// (max, sum, unnormalised output) partials in the workspace and the last CTA
// to finish it (atomic ticket, no waiting) merges them and writes the output.
//
// Semantics follow: "wavo 0.1.0, src/whisper/decoder.rs", Decoder::record_step
// (attend over pos+1 own rows and over all cross frames); "Nest whisper-tiny,
// src/lib.linnet", Attention.attend (scores scaled by rsqrt(D/Heads)) and
// DecoderLayer.step / .cross; "mlx-bun whisper.ts", #attention (precise
// softmax; beams share one broadcast encoder K/V); "transcribe.cpp,
// src/arch/qwen3_asr/decoder.h" (per-head Q/K RMSNorm, NeoX RoPE, GQA,
// StepBuildBatched: K/V written at row n_past, keys up to n_past attended).
#include <math.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "decode_attn.cuh"

namespace asrkv {

constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kRowsPerSlot = 2;

// In-place exclusive scan of data[0..n) over the whole block; data[n] gets
// the total.  tmp: 32 ints of shared memory.  All threads must call it.
__device__ void block_scan_excl(int* data, int n, int* tmp) {
  const int nt = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nw = (nt + 31) >> 5;
  const int chunk = (n + nt - 1) / nt;
  const int s = min(tid * chunk, n), e = min(s + chunk, n);
  int local = 0;
  for (int i = s; i < e; ++i) local += data[i];
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int v = lane < nw ? tmp[lane] : 0;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(kFull, inc, o);
      if (lane >= o) inc += t;
    }
    if (lane < nw) tmp[lane] = inc - v;
  }
  __syncthreads();
  int run = tmp[warp] + incl - local;
  for (int i = s; i < e; ++i) {
    const int v = data[i];
    data[i] = run;
    run += v;
  }
  if (s < e && e == n) data[n] = run;
  if (n == 0 && tid == 0) data[0] = 0;
  __syncthreads();
}

struct Tile {
  int g;       // source
  int row0;    // first row within the source
  int nr;      // rows in this tile
  bool first;  // first tile of this CTA's piece of source g
  bool last;   // last tile of this CTA's piece of source g
};

// Walks the tiles of the key range [k, k1) in order; the producer and the
// consumers run identical copies.
struct TileIter {
  const int* off;
  int S, tile_rows, g, prev_g;
  int64_t k, k1;
  __device__ TileIter(const int* off_, int S_, int64_t k0, int64_t k1_, int tr)
      : off(off_), S(S_), tile_rows(tr), g(0), prev_g(-1), k(k0), k1(k1_) {
    if (k0 < k1_) {
      int lo = 0, hi = S_;  // largest g < S with off[g] <= k0
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (off[mid] <= k0) lo = mid;
        else hi = mid;
      }
      g = lo;
    }
  }
  __device__ bool next(Tile& t) {
    if (k >= k1) return false;
    while (off[g + 1] <= k) ++g;
    const int64_t end = min((int64_t)off[g + 1], k1);
    const int nr = (int)min((int64_t)tile_rows, end - k);
    t.g = g;
    t.row0 = (int)(k - off[g]);
    t.nr = nr;
    t.first = g != prev_g;
    t.last = k + nr == end;
    prev_g = g;
    k += nr;
    return true;
  }
};

template <int HD>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = 1; o < HD / 8; o <<= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Per-head RMSNorm (weight * x * rsqrt(mean(x^2) + eps)) followed by NeoX
// RoPE on the 8 dims this lane holds (lane li of its group holds dims
// li*8 .. li*8+7).  Pair (i, i + HD/2) lives in lanes li and li ^ (G/2).
// rope: cos[HD/2] then sin[HD/2] for the current position.  Warp-uniform.
template <int HD>
__device__ __forceinline__ void norm_rope8(float* x, const float* __restrict__ w, float eps,
                                           const float* rope, int li) {
  constexpr int G = HD / 8;
  float ss = 0.f;
#pragma unroll
  for (int d = 0; d < 8; ++d) ss = fmaf(x[d], x[d], ss);
  ss = group_sum<HD>(ss);
  const float rinv = 1.0f / sqrtf(ss / (float)HD + eps);
  float xn[8];
#pragma unroll
  for (int d = 0; d < 8; ++d) xn[d] = w[li * 8 + d] * (x[d] * rinv);
  const bool lower = li < G / 2;
  const int i0 = (lower ? li : li - G / 2) * 8;
#pragma unroll
  for (int d = 0; d < 8; ++d) {
    const float partner = __shfl_xor_sync(kFull, xn[d], G / 2);
    const float c = rope[i0 + d], s = rope[HD / 2 + i0 + d];
    x[d] = lower ? (xn[d] * c - partner * s) : (xn[d] * c + partner * s);
  }
}

// cos/sin of p * theta_i for i < HD/2 into rope[] (consumer threads
// 0 .. HD/2-1).  The angle is formed and reduced modulo 2*pi in double; the
// reduced angle (|r| <= pi) is then evaluated in float.
template <int HD>
__device__ __forceinline__ void rope_table(float* rope, const double* theta, int p, int tid) {
  if (tid < HD / 2) {
    const double ang = (double)p * theta[tid];
    const double two_pi_hi = 6.283185307179586;       // 2*pi rounded to double
    const double two_pi_lo = 2.4492935982947064e-16;  // 2*pi - two_pi_hi
    const double kq = rint(ang * 0.15915494309189535);  // ang / (2*pi)
    double r = fma(-kq, two_pi_hi, ang);
    r = fma(-kq, two_pi_lo, r);
    float s, c;
    sincosf((float)r, &s, &c);
    rope[tid] = c;
    rope[HD / 2 + tid] = s;
  }
}

template <int HD, int NQ, int MAXT>
__global__ void __launch_bounds__(MAXT, 1) decode_attn_kernel(const __grid_constant__ DecodeArgs a) {
  constexpr int G = HD / 8;
  constexpr int RS = kRowsPerSlot;
  extern __shared__ __align__(128) unsigned char smem[];
  const DecodeSmem lay = decode_smem_layout(a.stages, a.n_src, a.R, a.Hkv, NQ, HD, a.stage_elems);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.bars);
  uint64_t* empty = full + a.stages;
  int* ctl = reinterpret_cast<int*>(smem + lay.ctl);  // [0] abort [1] ticket [2] unsorted
  int* off = reinterpret_cast<int*>(smem + lay.off);
  int* mst = reinterpret_cast<int*>(smem + lay.mstart);
  float* rope = reinterpret_cast<float*>(smem + lay.rope);
  float* merge = reinterpret_cast<float*>(smem + lay.merge);
  uint16_t* stage = reinterpret_cast<uint16_t*>(smem + lay.stage);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_cons = a.R * a.Hkv * G;  // a multiple of 32
  const int cons_warps = n_cons >> 5;
  const int S = a.n_src;
  const int qw = a.Hq * HD;

  if (tid == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], cons_warps);
    }
    for (int i = 0; i < 16; ++i) ctl[i] = 0;
    fence_barrier_init();
  }
  grid_dependency_wait();

  // ---- keys per source (off) and sequences per source (mst), then scans
  for (int g = tid; g <= S; g += blockDim.x) {
    off[g] = 0;
    mst[g] = 0;
  }
  __syncthreads();
  if (a.mode == kModeCross) {
    for (int b = tid; b < a.B; b += blockDim.x) {
      const int gr = a.group[b];
      if (gr >= 0 && gr < S) atomicAdd(&mst[gr], 1);
      if (b > 0 && a.group[b - 1] > gr) ctl[2] = 1;
    }
    __syncthreads();
    for (int g = tid; g < S; g += blockDim.x) off[g] = mst[g] > 0 ? a.fixed_len : 0;
  } else {
    for (int g = tid; g < S; g += blockDim.x) {
      const int v = a.lens[g];
      int keys;
      if (a.mode == kModeSelf) keys = (v >= 1 && v <= a.capacity) ? v : 0;
      else keys = (v >= 0 && v < a.capacity) ? v : 0;  // rows cached before the new one
      off[g] = keys;
      mst[g] = 1;
    }
  }
  __syncthreads();
  block_scan_excl(off, S, reinterpret_cast<int*>(rope));
  block_scan_excl(mst, S, reinterpret_cast<int*>(rope));
  const bool unsorted = a.mode == kModeCross && ctl[2] != 0;

  // ---- CTA 0 zeroes the outputs of sequences that are skipped
  if (blockIdx.x == 0) {
    for (int b = warp; b < a.B; b += blockDim.x >> 5) {
      int bad = 0;
      if (unsorted) {
        bad = ASR_DEVERR_INDEX;
      } else if (a.mode == kModeCross) {
        const int gr = a.group[b];
        if (gr < 0 || gr >= S) bad = ASR_DEVERR_INDEX;
        else if (b - mst[gr] >= a.max_members) bad = ASR_DEVERR_BEAMS;
      } else {
        const int v = a.lens[b];
        const bool ok =
            a.mode == kModeSelf ? (v >= 1 && v <= a.capacity) : (v >= 0 && v < a.capacity);
        if (!ok) bad = ASR_DEVERR_LEN;
      }
      if (bad) {
        for (int i = lane * 4; i < qw; i += 128)
          *reinterpret_cast<float4*>(a.out + (int64_t)b * qw + i) = make_float4(0.f, 0.f, 0.f, 0.f);
        if (lane == 0) set_dev_err(a.dev_err, bad);
      }
    }
  }
  if (unsorted) {
    grid_launch_dependents();
    return;
  }

  // ---- this CTA's share of the flattened key axis
  const int64_t total = off[S];
  const int P = gridDim.x;
  int64_t share = (total + P - 1) / P;
  if (share < a.tile_rows) share = a.tile_rows;
  const int64_t k0 = (int64_t)blockIdx.x * share;
  const int64_t k1 = min(k0 + share, total);

  if (warp == cons_warps) {
    // ======================= producer warp: one lane issues bulk copies
    if (lane == 0 && k0 < k1) {
      const uint64_t pol = policy_evict_first();
      TileIter it(off, S, k0, k1, a.tile_rows);
      Tile tl;
      for (int t = 0; it.next(tl); ++t) {
        const int s = t % a.stages;
        if (t >= a.stages && !mbar_wait(&empty[s], ((t / a.stages) - 1) & 1)) {
          set_dev_err(a.dev_err, ASR_DEVERR_TIMEOUT);
          ctl[0] = 1;
          break;
        }
        const uint32_t bytes = (uint32_t)tl.nr * (uint32_t)a.row_elems * 2u;
        mbar_arrive_expect_tx(&full[s], bytes);
        bulk_g2s(stage + (size_t)s * a.stage_elems,
                 a.kv + (int64_t)tl.g * a.src_stride + (int64_t)tl.row0 * a.row_elems, bytes,
                 &full[s], pol);
      }
    }
    grid_launch_dependents();
    return;
  }
  if (warp > cons_warps) return;

  // ======================= consumers
  const int grp = tid / G, li = tid % G;
  const int h = grp % a.Hkv, r = grp / a.Hkv;
  const int rep = a.rep;

  float qv[NQ][8], o[NQ][8], m[NQ], l[NQ];
  int nq = 0, mbase = 0;
  // New-token K/V of the GQA step (f16-rounded, as floats) and its scores.
  float kn[8], vn[8], snew[NQ];
#pragma unroll
  for (int d = 0; d < 8; ++d) kn[d] = vn[d] = 0.f;
#pragma unroll
  for (int qi = 0; qi < NQ; ++qi) snew[qi] = 0.f;

  auto seg_begin = [&](int g) {
    const int cnt = mst[g + 1] - mst[g];
    mbase = mst[g];
    nq = min(cnt, a.max_members) * rep;
    if (a.mode == kModeGqa) {
      named_bar(1, n_cons);
      rope_table<HD>(rope, a.theta, a.lens[g], tid);
      named_bar(1, n_cons);
    }
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) {
      m[qi] = -INFINITY;
      l[qi] = 0.f;
#pragma unroll
      for (int d = 0; d < 8; ++d) o[qi][d] = 0.f;
      if (qi < nq) {
        const int b = mbase + qi / rep;
        const int hq = h * rep + qi % rep;
        const float* src = a.q + (int64_t)b * a.q_stride + hq * HD + li * 8;
        const float4 x0 = *reinterpret_cast<const float4*>(src);
        const float4 x1 = *reinterpret_cast<const float4*>(src + 4);
        float x[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        if (a.mode == kModeGqa) norm_rope8<HD>(x, a.wq, a.eps, rope, li);
#pragma unroll
        for (int d = 0; d < 8; ++d) qv[qi][d] = x[d] * a.qscale;
      } else {
#pragma unroll
        for (int d = 0; d < 8; ++d) qv[qi][d] = 0.f;
      }
    }
  };

  // Fold the new token (GQA) into (M, Ls, O) and write the normalised
  // output of query qi.  Contains no shuffles: callable per group.
  auto finalize = [&](int qi, float M, float Ls, float* O) {
    if (a.mode == kModeGqa) {
      const float mn = fmaxf(M, snew[qi]);
      const float ca = exp2f(M - mn), cb = exp2f(snew[qi] - mn);
      Ls = Ls * ca + cb;
#pragma unroll
      for (int d = 0; d < 8; ++d) O[d] = fmaf(cb, vn[d], O[d] * ca);
    }
    const int b = mbase + qi / rep;
    const int hq = h * rep + qi % rep;
    const float inv = 1.0f / Ls;
    float* dst = a.out + (int64_t)b * qw + hq * HD + li * 8;
    *reinterpret_cast<float4*>(dst) = make_float4(O[0] * inv, O[1] * inv, O[2] * inv, O[3] * inv);
    *reinterpret_cast<float4*>(dst + 4) =
        make_float4(O[4] * inv, O[5] * inv, O[6] * inv, O[7] * inv);
  };

  auto seg_end = [&](int g) {
    // GQA: the new token's key/value, computed by every group (warp-uniform
    // code: it shuffles), appended to the cache by row slot 0.
    if (a.mode == kModeGqa) {
      const int p = a.lens[g];
      const float* ks = a.k_new + (int64_t)g * a.Hkv * HD + h * HD + li * 8;
      const float* vs = a.v_new + (int64_t)g * a.Hkv * HD + h * HD + li * 8;
      const float4 x0 = *reinterpret_cast<const float4*>(ks);
      const float4 x1 = *reinterpret_cast<const float4*>(ks + 4);
      const float4 v0 = *reinterpret_cast<const float4*>(vs);
      const float4 v1 = *reinterpret_cast<const float4*>(vs + 4);
      float x[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      float vv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      norm_rope8<HD>(x, a.wk, a.eps, rope, li);
      const uint4 kh = f8_to_h8(x);
      const uint4 vh = f8_to_h8(vv);
      h8_to_f8(kh, kn);
      h8_to_f8(vh, vn);
      if (r == 0) {
        uint16_t* row = a.cache_w + (int64_t)g * a.src_stride + (int64_t)p * a.row_elems;
        *reinterpret_cast<uint4*>(row + h * HD + li * 8) = kh;
        *reinterpret_cast<uint4*>(row + a.Hkv * HD + h * HD + li * 8) = vh;
      }
#pragma unroll
      for (int qi = 0; qi < NQ; ++qi) {
        if (qi < nq) {
          float sdot = 0.f;
#pragma unroll
          for (int d = 0; d < 8; ++d) sdot = fmaf(qv[qi][d], kn[d], sdot);
          snew[qi] = group_sum<HD>(sdot);
        }
      }
    }
    // merge the row slots of each head into slot 0
    named_bar(1, n_cons);
    if (r > 0) {
#pragma unroll
      for (int qi = 0; qi < NQ; ++qi) {
        if (qi < nq) {
          float* mb = merge + (((r - 1) * a.Hkv + h) * NQ + qi) * (HD + 2);
#pragma unroll
          for (int d = 0; d < 8; ++d) mb[li * 8 + d] = o[qi][d];
          if (li == 0) {
            mb[HD] = m[qi];
            mb[HD + 1] = l[qi];
          }
        }
      }
    }
    named_bar(1, n_cons);
    if (r == 0) {
      for (int r2 = 1; r2 < a.R; ++r2) {
#pragma unroll
        for (int qi = 0; qi < NQ; ++qi) {
          if (qi < nq) {
            const float* mb = merge + (((r2 - 1) * a.Hkv + h) * NQ + qi) * (HD + 2);
            const float m2 = mb[HD], l2 = mb[HD + 1];
            const float mn = fmaxf(m[qi], m2);
            if (mn != -INFINITY) {
              const float ca = exp2f(m[qi] - mn), cb = exp2f(m2 - mn);
              l[qi] = l[qi] * ca + l2 * cb;
#pragma unroll
              for (int d = 0; d < 8; ++d) o[qi][d] = fmaf(cb, mb[li * 8 + d], o[qi][d] * ca);
              m[qi] = mn;
            }
          }
        }
      }
    }
    // pieces of this source over the grid
    const int64_t go = off[g], gl = (int64_t)off[g + 1] - off[g];
    const int first = gl > 0 ? (int)(go / share) : 0;
    const int lastp = gl > 0 ? (int)((go + gl - 1) / share) : 0;
    const int parts = gl > 0 ? lastp - first + 1 : 0;
    if (parts <= 1) {
      if (r == 0) {
#pragma unroll
        for (int qi = 0; qi < NQ; ++qi)
          if (qi < nq) finalize(qi, m[qi], l[qi], o[qi]);
      }
      return;
    }
    if (r == 0) {
      const int64_t slot = (int64_t)blockIdx.x + g;
#pragma unroll
      for (int qi = 0; qi < NQ; ++qi) {
        if (qi < nq) {
          const int64_t pidx = (slot * a.max_members + qi / rep) * a.Hq + h * rep + qi % rep;
          float* po = a.part_o + pidx * HD + li * 8;
          *reinterpret_cast<float4*>(po) = make_float4(o[qi][0], o[qi][1], o[qi][2], o[qi][3]);
          *reinterpret_cast<float4*>(po + 4) = make_float4(o[qi][4], o[qi][5], o[qi][6], o[qi][7]);
          if (li == 0) *reinterpret_cast<float2*>(a.part_ml + pidx * 2) = make_float2(m[qi], l[qi]);
        }
      }
      __threadfence();
    }
    named_bar(1, n_cons);
    if (tid == 0) {
      const int old = atomicAdd(&a.counters[g], 1);
      const int is_last = old == parts - 1;
      if (is_last) atomicExch(&a.counters[g], 0);
      ctl[1] = is_last;
    }
    named_bar(1, n_cons);
    if (ctl[1]) {
      __threadfence();
      for (int qi = r; qi < nq; qi += a.R) {
        float M = -INFINITY, Ls = 0.f, O[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int kp = first; kp <= lastp; ++kp) {
          const int64_t slot = (int64_t)kp + g;
          const int64_t pidx = (slot * a.max_members + qi / rep) * a.Hq + h * rep + qi % rep;
          const float2 ml = __ldcg(reinterpret_cast<const float2*>(a.part_ml + pidx * 2));
          const float4 p0 = ld_cg_f4(a.part_o + pidx * HD + li * 8);
          const float4 p1 = ld_cg_f4(a.part_o + pidx * HD + li * 8 + 4);
          const float mn = fmaxf(M, ml.x);
          if (mn == -INFINITY) continue;
          const float ca = exp2f(M - mn), cb = exp2f(ml.x - mn);
          Ls = Ls * ca + ml.y * cb;
          const float pv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
          for (int d = 0; d < 8; ++d) O[d] = fmaf(cb, pv[d], O[d] * ca);
          M = mn;
        }
        finalize(qi, M, Ls, O);
      }
    }
  };

  if (k0 < k1) {
    TileIter it(off, S, k0, k1, a.tile_rows);
    Tile tl;
    for (int t = 0; it.next(tl); ++t) {
      if (tl.first) seg_begin(tl.g);
      const int s = t % a.stages;
      if (!mbar_wait(&full[s], (t / a.stages) & 1)) {
        set_dev_err(a.dev_err, ASR_DEVERR_TIMEOUT);
        break;
      }
      const uint16_t* tb = stage + (size_t)s * a.stage_elems;
      float kf[RS][8], vf[RS][8];
      bool val[RS];
#pragma unroll
      for (int i = 0; i < RS; ++i) {
        const int row = r + i * a.R;
        val[i] = row < tl.nr;
        if (val[i]) {
          const uint16_t* rp = tb + row * a.row_elems + h * HD + li * 8;
          const uint4 ku = *reinterpret_cast<const uint4*>(rp);
          const uint4 vu = *reinterpret_cast<const uint4*>(rp + a.Hkv * HD);
          h8_to_f8(ku, kf[i]);
          h8_to_f8(vu, vf[i]);
        } else {
#pragma unroll
          for (int d = 0; d < 8; ++d) kf[i][d] = vf[i][d] = 0.f;
        }
      }
      // the stage is in registers now: hand it back to the producer
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll
      for (int qi = 0; qi < NQ; ++qi) {
        if (qi < nq) {
          float sc[RS];
#pragma unroll
          for (int i = 0; i < RS; ++i) {
            float dsum = 0.f;
#pragma unroll
            for (int d = 0; d < 8; ++d) dsum = fmaf(qv[qi][d], kf[i][d], dsum);
            sc[i] = dsum;
          }
#pragma unroll
          for (int o2 = 1; o2 < G; o2 <<= 1) {
#pragma unroll
            for (int i = 0; i < RS; ++i) sc[i] += __shfl_xor_sync(kFull, sc[i], o2);
          }
          float mt = -INFINITY;
#pragma unroll
          for (int i = 0; i < RS; ++i)
            if (val[i]) mt = fmaxf(mt, sc[i]);
          if (mt != -INFINITY) {
            const float mn = fmaxf(m[qi], mt);
            const float alpha = exp2f(m[qi] - mn);
            float p[RS], psum = 0.f;
#pragma unroll
            for (int i = 0; i < RS; ++i) {
              p[i] = val[i] ? exp2f(sc[i] - mn) : 0.f;
              psum += p[i];
            }
            l[qi] = fmaf(l[qi], alpha, psum);
#pragma unroll
            for (int d = 0; d < 8; ++d) {
              float acc = o[qi][d] * alpha;
#pragma unroll
              for (int i = 0; i < RS; ++i) acc = fmaf(p[i], vf[i][d], acc);
              o[qi][d] = acc;
            }
            m[qi] = mn;
          }
        }
      }
      if (tl.last) seg_end(tl.g);
    }
  }

  // GQA sources with no cached rows (n_past == 0): only the new token; CTA
  // g % P handles source g.
  if (a.mode == kModeGqa) {
    for (int g = blockIdx.x; g < S; g += P) {
      if (a.lens[g] == 0) {
        seg_begin(g);
        seg_end(g);
      }
    }
  }
  grid_launch_dependents();
}

// ---------------------------------------------------------------- host ----

struct DecodePlan {
  int R, tile_rows, stages, stage_elems, threads, smem, grid;
};

static int max_threads_for(int NQ) { return NQ <= 2 ? 640 : (NQ <= 4 ? 512 : 256); }

template <int HD, int NQ>
static void* kernel_ptr() {
  return (void*)decode_attn_kernel<HD, NQ, (NQ <= 2 ? 640 : (NQ <= 4 ? 512 : 256))>;
}

static int nq_bucket(int nq) {
  if (nq <= 1) return 1;
  if (nq <= 2) return 2;
  if (nq <= 4) return 4;
  if (nq <= 8) return 8;
  return 0;
}

static void* kernel_for(int HD, int NQ) {
  if (HD == 64) {
    switch (NQ) {
      case 1: return kernel_ptr<64, 1>();
      case 2: return kernel_ptr<64, 2>();
      case 4: return kernel_ptr<64, 4>();
      case 8: return kernel_ptr<64, 8>();
    }
  } else if (HD == 128) {
    switch (NQ) {
      case 1: return kernel_ptr<128, 1>();
      case 2: return kernel_ptr<128, 2>();
      case 4: return kernel_ptr<128, 4>();
      case 8: return kernel_ptr<128, 8>();
    }
  }
  return nullptr;
}

// Row slots R: as many as fit the thread budget (at most 512 consumer
// threads), with the consumer count a multiple of 32.  Stages: as many as fit
// 200 KB of shared memory, 2..8.
static bool plan_decode(int HD, int NQ, int Hkv, int row_elems, int n_src, DecodePlan& p) {
  const int G = HD / 8;
  const int per_slot = Hkv * G;
  const int budget = std::min(max_threads_for(NQ) - 32, 512);
  int best = 0;
  for (int R = 1; R * per_slot <= budget; ++R)
    if ((R * per_slot) % 32 == 0) best = R;
  if (best == 0) return false;
  p.R = best;
  p.threads = best * per_slot + 32;
  p.tile_rows = best * kRowsPerSlot;
  p.stage_elems = dsm_align(p.tile_rows * row_elems, 64);
  const int smem_cap = 200 * 1024;
  int stages = 8;
  while (stages > 2 &&
         decode_smem_layout(stages, n_src, p.R, Hkv, NQ, HD, p.stage_elems).total > smem_cap)
    --stages;
  p.stages = stages;
  p.smem = decode_smem_layout(stages, n_src, p.R, Hkv, NQ, HD, p.stage_elems).total;
  if (p.smem > 227 * 1024) return false;
  return true;
}

size_t decode_ws_bytes(int n_src, int max_members, int Hq, int HD, int sms) {
  const int64_t slots = (int64_t)kMaxCtasPerSm * sms + n_src;
  const size_t counters = align_up((size_t)n_src * 4, 256);
  const size_t ml = align_up((size_t)slots * max_members * Hq * 2 * 4, 256);
  const size_t o = (size_t)slots * max_members * Hq * HD * 4;
  return counters + ml + o;
}

static std::once_flag g_attr_once[2][4];

static int launch_decode(DecodeArgs& a, int HD, int nq_needed, void* ws, size_t ws_bytes,
                         cudaStream_t stream) {
  const int NQ = nq_bucket(nq_needed);
  if (NQ == 0) return ASR_ERR_UNSUPPORTED;
  DecodePlan p;
  if (!plan_decode(HD, NQ, a.Hkv, a.row_elems, a.n_src, p)) return ASR_ERR_UNSUPPORTED;
  const int sms = device_sm_count();
  if (sms <= 0) return ASR_ERR_CUDA;
  const size_t need = decode_ws_bytes(a.n_src, a.max_members, a.Hq, HD, sms);
  if (!ws || ((uintptr_t)ws & 255u) != 0 || ws_bytes < need) return ASR_ERR_WORKSPACE;
  void* fn = kernel_for(HD, NQ);
  const int hi = HD == 64 ? 0 : 1;
  const int ni = NQ == 1 ? 0 : NQ == 2 ? 1 : NQ == 4 ? 2 : 3;
  cudaError_t attr_err = cudaSuccess;
  std::call_once(g_attr_once[hi][ni], [&] {
    attr_err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
  });
  if (attr_err != cudaSuccess) return ASR_ERR_CUDA;
  int occ = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, p.threads, p.smem) != cudaSuccess)
    return ASR_ERR_CUDA;
  occ = std::max(1, std::min(occ, kMaxCtasPerSm));
  p.grid = sms * occ;
  char* w = static_cast<char*>(ws);
  a.counters = reinterpret_cast<int*>(w);
  w += align_up((size_t)a.n_src * 4, 256);
  const int64_t slots = (int64_t)kMaxCtasPerSm * sms + a.n_src;
  a.part_ml = reinterpret_cast<float*>(w);
  w += align_up((size_t)slots * a.max_members * a.Hq * 2 * 4, 256);
  a.part_o = reinterpret_cast<float*>(w);
  a.R = p.R;
  a.tile_rows = p.tile_rows;
  a.stages = p.stages;
  a.stage_elems = p.stage_elems;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(p.threads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* params[] = {&a};
  cudaError_t e = cudaLaunchKernelExC(&cfg, fn, params);
  return e == cudaSuccess ? ASR_OK : ASR_ERR_CUDA;
}

static bool rows_fit_int(int64_t n_src, int64_t rows) { return n_src * rows < (1LL << 31); }

}  // namespace asrkv

using namespace asrkv;

extern "C" int asr_self_attn_step(const float* q, int64_t q_stride, const uint16_t* cache,
                                  int64_t seq_stride, const int32_t* lens, int B, int heads,
                                  int head_dim, int capacity, float scale, float* out, void* ws,
                                  size_t ws_bytes, int32_t* dev_err, asr_stream_t stream) {
  if (B < 0 || B > ASR_MAX_BATCH || heads < 1 || capacity < 1) return ASR_ERR_INVALID_ARG;
  if ((head_dim != 64 && head_dim != 128) || heads > ASR_MAX_KV_HEADS) return ASR_ERR_UNSUPPORTED;
  if (B == 0) return ASR_OK;
  if (!q || !cache || !lens || !out) return ASR_ERR_INVALID_ARG;
  const int64_t row = 2LL * heads * head_dim;
  if (q_stride < (int64_t)heads * head_dim || seq_stride < (int64_t)capacity * row)
    return ASR_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(cache) || !aligned16(out) || q_stride % 4 != 0 ||
      seq_stride % 8 != 0)
    return ASR_ERR_MISALIGNED;
  if (!rows_fit_int(B, capacity)) return ASR_ERR_UNSUPPORTED;
  DecodeArgs a = {};
  a.q = q;
  a.q_stride = q_stride;
  a.kv = cache;
  a.src_stride = seq_stride;
  a.row_elems = (int)row;
  a.n_src = B;
  a.B = B;
  a.lens = lens;
  a.capacity = capacity;
  a.Hq = heads;
  a.Hkv = heads;
  a.rep = 1;
  a.max_members = 1;
  a.qscale = scale * kLog2e;
  a.out = out;
  a.dev_err = dev_err;
  a.mode = kModeSelf;
  return launch_decode(a, head_dim, 1, ws, ws_bytes, (cudaStream_t)stream);
}

extern "C" int asr_cross_attn_step(const float* q, int64_t q_stride, const uint16_t* cross,
                                   int64_t group_stride, const int32_t* group, int B, int G,
                                   int max_beams, int heads, int head_dim, int frames, float scale,
                                   float* out, void* ws, size_t ws_bytes, int32_t* dev_err,
                                   asr_stream_t stream) {
  if (B < 0 || B > ASR_MAX_BATCH || G < 1 || G > ASR_MAX_BATCH || heads < 1 || frames < 1 ||
      max_beams < 1)
    return ASR_ERR_INVALID_ARG;
  if ((head_dim != 64 && head_dim != 128) || heads > ASR_MAX_KV_HEADS || max_beams > ASR_MAX_BEAMS)
    return ASR_ERR_UNSUPPORTED;
  if (B == 0) return ASR_OK;
  if (!q || !cross || !group || !out) return ASR_ERR_INVALID_ARG;
  const int64_t row = 2LL * heads * head_dim;
  if (q_stride < (int64_t)heads * head_dim || group_stride < (int64_t)frames * row)
    return ASR_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(cross) || !aligned16(out) || q_stride % 4 != 0 ||
      group_stride % 8 != 0)
    return ASR_ERR_MISALIGNED;
  if (!rows_fit_int(G, frames)) return ASR_ERR_UNSUPPORTED;
  DecodeArgs a = {};
  a.q = q;
  a.q_stride = q_stride;
  a.kv = cross;
  a.src_stride = group_stride;
  a.row_elems = (int)row;
  a.n_src = G;
  a.B = B;
  a.group = group;
  a.fixed_len = frames;
  a.Hq = heads;
  a.Hkv = heads;
  a.rep = 1;
  a.max_members = max_beams;
  a.qscale = scale * kLog2e;
  a.out = out;
  a.dev_err = dev_err;
  a.mode = kModeCross;
  return launch_decode(a, head_dim, max_beams, ws, ws_bytes, (cudaStream_t)stream);
}

extern "C" int asr_gqa_step(const float* q, const float* k_new, const float* v_new,
                            const float* q_norm_w, const float* k_norm_w, float eps,
                            float rope_base, const int32_t* n_past, uint16_t* cache,
                            int64_t seq_stride, int capacity, int B, int q_heads, int kv_heads,
                            int head_dim, float scale, float* out, void* ws, size_t ws_bytes,
                            int32_t* dev_err, asr_stream_t stream) {
  if (B < 0 || B > ASR_MAX_BATCH || q_heads < 1 || kv_heads < 1 || capacity < 1 ||
      !(eps >= 0.f) || !(rope_base > 0.f))
    return ASR_ERR_INVALID_ARG;
  if ((head_dim != 64 && head_dim != 128) || kv_heads > ASR_MAX_KV_HEADS ||
      q_heads % kv_heads != 0 || q_heads / kv_heads > ASR_MAX_BEAMS)
    return ASR_ERR_UNSUPPORTED;
  if (B == 0) return ASR_OK;
  if (!q || !k_new || !v_new || !q_norm_w || !k_norm_w || !n_past || !cache || !out)
    return ASR_ERR_INVALID_ARG;
  const int64_t row = 2LL * kv_heads * head_dim;
  if (seq_stride < (int64_t)capacity * row) return ASR_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(q_norm_w) ||
      !aligned16(k_norm_w) || !aligned16(cache) || !aligned16(out) || seq_stride % 8 != 0)
    return ASR_ERR_MISALIGNED;
  if (!rows_fit_int(B, capacity)) return ASR_ERR_UNSUPPORTED;
  DecodeArgs a = {};
  a.q = q;
  a.q_stride = (int64_t)q_heads * head_dim;
  a.kv = cache;
  a.cache_w = cache;
  a.src_stride = seq_stride;
  a.row_elems = (int)row;
  a.n_src = B;
  a.B = B;
  a.lens = n_past;
  a.capacity = capacity;
  a.Hq = q_heads;
  a.Hkv = kv_heads;
  a.rep = q_heads / kv_heads;
  a.max_members = 1;
  a.qscale = scale * kLog2e;
  a.out = out;
  a.dev_err = dev_err;
  a.mode = kModeGqa;
  a.k_new = k_new;
  a.v_new = v_new;
  a.wq = q_norm_w;
  a.wk = k_norm_w;
  a.eps = eps;
  for (int i = 0; i < head_dim / 2; ++i) a.theta[i] = pow((double)rope_base, -2.0 * i / head_dim);
  return launch_decode(a, head_dim, a.rep, ws, ws_bytes, (cudaStream_t)stream);
}
