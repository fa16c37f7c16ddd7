// decode_attn.cu -- one-token attention over f16 K/V caches (a2, a3, a4, a5).
//
// Method: split-K flash-decoding with a log-sum-exp combine.  The work of a
// call is cut into units: a unit is one source (the sequence for
// self-attention and the GQA step, the beam group for cross-attention) and
// one group of hs of its KV heads (HS = Hkv / hs groups per source; HS = 1
// when the sources are short next to a CTA's share).  Every (unit, key)
// pair lies on one flattened key axis and a persistent grid of P CTAs takes
// equal contiguous shares of it, so variable lengths stay balanced to within
// one tile.  A CTA streams its share as tiles of cache rows into a
// multi-stage shared-memory ring (mbarrier full/empty pairs, one producer
// warp): whole rows with one bulk TMA copy per tile when HS = 1, else the
// unit's K and V chunks of each row through a 5-D tensor map.  The consumer
// threads form groups of G = HD/DPL lanes (DPL = 16 dims per lane for one or
// two queries, 8 for four or eight); a group owns one KV head of the unit,
// keeps its queries (beams of the group x query heads of the KV head) in
// registers, and runs an online softmax in the log2 domain over the rows it
// is given.  At the end of a unit's piece the row slots are merged in shared
// memory (a tree); a unit split over several CTAs leaves (max, sum,
// unnormalised output) partials in the workspace and the last CTA to finish
// it (atomic ticket, no waiting) merges them and writes the output.  Cutting
// a long source into head groups divides both the number of partials of a
// unit and the query heads each holds, so that last merge stays short.
//
// Semantics follow: "wavo 0.1.0, src/whisper/decoder.rs", Decoder::record_step
// (attend over pos+1 own rows and over all cross frames); "Nest whisper-tiny,
// src/lib.linnet", Attention.attend (scores scaled by rsqrt(D/Heads)) and
// DecoderLayer.step / .cross; "mlx-bun whisper.ts", #attention (precise
// softmax; beams share one broadcast encoder K/V); "transcribe.cpp,
// src/arch/qwen3_asr/decoder.h" (per-head Q/K RMSNorm, NeoX RoPE, GQA,
// StepBuildBatched: K/V written at row n_past, keys up to n_past attended).
#include <math.h>
#include <stdio.h>
#include <stdlib.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "decode_attn.cuh"
#include "tcgen05.cuh"

namespace asrkv {

constexpr float kLog2e = 1.4426950408889634f;
// Merges a CTA defers to the end of its tiles.  Only a unit that crosses an
// end of the CTA's share has pieces in other CTAs, so a CTA takes at most two
// tickets per launch.
constexpr int kMergeList = 2;
constexpr unsigned kFull = 0xffffffffu;

// History rows of one self / GQA source that the call streams, from its
// length entry (0 for an out-of-range entry).  Self: keys including the new
// token, less the appended one; GQA: n_past, the rows cached before the new
// token.
__device__ __forceinline__ int streamed_rows(const DecodeArgs& a, int v) {
  if (a.mode == kModeSelf) return (v >= 1 && v <= a.capacity) ? v - a.append : 0;
  return (v >= 0 && v < a.capacity) ? v : 0;
}

// Offsets of the sources on the flattened key axis, computed by one warp:
// off[g] = HS * sum over g' < g of (virtual rows + streamed rows of g'),
// off[S] = the total (returned).  A source with nothing to stream takes no
// room.  Cross: a group is streamed when some sequence belongs to it (the
// flags go through off[] itself, which is then scanned in place); returns -1
// when the group indices are not sorted.  cg: read the inputs from L2 only
// (the early, hint-only pass before the grid dependency wait).  With a beam
// reorder, source g takes the length of sequence idx[g] (0, nothing to
// stream, for an index outside [0, S)) and src_out[g] receives idx[g].
__device__ int warp_offsets(const DecodeArgs& a, int* off, int S, int lane, bool cg,
                             int* lens_out = nullptr, int* src_out = nullptr) {
  if (a.mode == kModeCross) {
    for (int g = lane; g <= S; g += 32) off[g] = 0;
    __syncwarp();
    bool unsorted = false;
    for (int b = lane; b < a.B; b += 32) {
      const int gr = cg ? __ldcg(a.group + b) : a.group[b];
      if (b > 0 && (cg ? __ldcg(a.group + b - 1) : a.group[b - 1]) > gr) unsorted = true;
      if (gr >= 0 && gr < S) off[gr] = 1;  // every writer stores the same value
    }
    if (__any_sync(kFull, unsorted)) return -1;
    __syncwarp();
  }
  int run = 0;
  for (int base = 0; base < S; base += 32) {
    const int g = base + lane;
    int keys = 0;
    if (g < S) {
      if (a.mode == kModeCross) {
        keys = off[g] ? a.HS * (a.fixed_len + a.seg_rows) : 0;
      } else {
        int v;
        if (a.idx) {
          const int sq = cg ? __ldcg(a.idx + g) : a.idx[g];
          v = (sq >= 0 && sq < S) ? (cg ? __ldcg(a.lens + sq) : a.lens[sq]) : 0;
          if (src_out) src_out[g] = sq;
        } else {
          v = cg ? __ldcg(a.lens + g) : a.lens[g];
        }
        if (lens_out) lens_out[g] = v;
        const int k = streamed_rows(a, v);
        keys = k > 0 ? a.HS * (k + a.seg_rows) : 0;
      }
    }
    int incl = keys;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += t;
    }
    __syncwarp();
    if (g < S) off[g] = run + incl - keys;
    run += __shfl_sync(kFull, incl, 31);
  }
  if (lane == 0) off[S] = run;
  __syncwarp();
  return run;
}

struct Tile {
  int u;       // unit (source g, head group hg): u = g * HS + hg
  int g, hg;
  int row0;    // first row within the source
  int nr;      // rows in this tile
  bool first;  // first tile of this CTA's piece of unit u
  bool last;   // last tile of this CTA's piece of unit u
};

// Where unit u lies on the flattened axis: its first real row go and its
// real rows gl (gl <= 0: the unit streams nothing).  Each unit of a source
// spans the same length: vrows virtual rows (never loaded; they charge the
// CTA that enters the unit for its per-unit work) then the source's rows.
// The axis fits in int (checked on the host), so 32-bit arithmetic serves.
struct UnitSpan {
  int go, gl;
};
__device__ __forceinline__ UnitSpan unit_span(const int* off, int HS, int vrows, int u) {
  const int g = HS == 1 ? u : u / HS, hg = u - g * HS;
  const int base = off[g];
  const int len = HS == 1 ? off[g + 1] - base : (off[g + 1] - base) / HS;
  return {base + hg * len + vrows, len - vrows};
}

// Cross: the first sequence of each group.  The groups are sorted, so the
// first sequence of group g is the first b with group[b] >= g: sequence b
// (with group[-1] = -1 and group[B] = S, values clamped into [-1, S]) sets
// m[g] = b for every g in (group[b-1], group[b]].  Threads t, t + nt, ...
__device__ __forceinline__ void first_members(const DecodeArgs& a, int* m, int S, int t, int nt) {
  for (int b = t; b <= a.B; b += nt) {
    const int cur = b < a.B ? min(max(a.group[b], -1), S) : S;
    const int prev = b > 0 ? min(max(a.group[b - 1], -1), S) : -1;
    for (int g = prev + 1; g <= cur; ++g) m[g] = b;
  }
}

// Does CTA c hold the first real row of unit u?  That CTA folds the new
// token in (append).  A unit with no cached rows is folded by the CTA that
// handles it alone.
__device__ __forceinline__ bool owns_first_row(const int* off, int HS, int vrows, int share, int u,
                                               int c) {
  const UnitSpan sp = unit_span(off, HS, vrows, u);
  return sp.gl <= 0 || sp.go / share == c;
}

// Walks the tiles of the key range [k, k1) in order; the producer and the
// consumers run identical copies.  It steps from unit to unit without
// dividing (one division places the start).
struct TileIter {
  const int* off;
  int S, HS, tile_rows, vrows;
  int g, hg, ustart, len, prev_u;
  int k, k1;
  __device__ TileIter(const int* off_, int S_, int HS_, int k0, int k1_, int tr, int vr)
      : off(off_), S(S_), HS(HS_), tile_rows(tr), vrows(vr), g(0), hg(0), ustart(0), len(0),
        prev_u(-1), k(k0), k1(k1_) {
    if (k0 < k1_) {
      int lo = 0, hi = S_;  // largest g < S with off[g] <= k0
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (off[mid] <= k0) lo = mid;
        else hi = mid;
      }
      while (off[lo + 1] <= k0) ++lo;  // skip sources that take no room
      g = lo;
      len = HS == 1 ? off[g + 1] - off[g] : (off[g + 1] - off[g]) / HS;
      hg = HS == 1 ? 0 : (k0 - off[g]) / len;
      ustart = off[g] + hg * len;
    }
  }
  __device__ bool next(Tile& t) {
    if (k >= k1) return false;
    while (k >= ustart + len) {  // the next unit: same source, else the next source with room
      if (++hg == HS) {
        hg = 0;
        do {
          ++g;
        } while (off[g + 1] == off[g]);
        len = HS == 1 ? off[g + 1] - off[g] : (off[g + 1] - off[g]) / HS;
        ustart = off[g];
      } else {
        ustart += len;
      }
    }
    const int real0 = ustart + vrows;  // < ustart + len: a unit has a real row
    if (k < real0) {
      k = real0;
      if (k >= k1) return false;
    }
    const int end = min(ustart + len, k1);
    const int nr = min(tile_rows, end - k);
    t.g = g;
    t.hg = hg;
    t.u = g * HS + hg;
    t.row0 = k - real0;
    t.nr = nr;
    t.first = t.u != prev_u;
    t.last = k + nr == end;
    prev_u = t.u;
    k += nr;
    return true;
  }
};

// Tiled 5-D TMA load of one box into shared memory, completing its bytes on
// bar, with an L2 cache policy.  c0 (innermost) is always 0 here.
__device__ __forceinline__ void tma_load_5d(void* dst, const CUtensorMap* map, int c1, int c2,
                                            int c3, int c4, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
      "r"(smem_addr(bar)), "l"(pol)
      : "memory");
}

// Hint: bring one box of a 5-D tensor into L2 (writes nothing, completes
// nothing).
__device__ __forceinline__ void tma_prefetch_5d(const CUtensorMap* map, int c1, int c2, int c3,
                                                int c4) {
  asm volatile("cp.async.bulk.prefetch.tensor.5d.L2.global.tile [%0, {%1, %2, %3, %4, %5}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
               : "memory");
}

// ---- packed fp32 pairs and the fast base-2 exponential ---------------------

// 2^x with the hardware approximation (relative error ~2^-22; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 8 f16 held in registers -> 4 float pairs.  Takes the vector by value: a
// reference into shared memory would make the conversion re-read it as four
// 32-bit loads.
__device__ __forceinline__ void h8_to_f2x4(const uint4 u, float2* f) {
  const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) f[i] = __half22float2(h[i]);
}

template <int G>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = 1; o < G; o <<= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Lane layout of one head vector: a group of G = HD/DPL lanes covers the
// head; lane li holds NCH = DPL/8 chunks of 8 dims.  Register slot j holds
// chunk li + (j ^ sw)*G, i.e. dims (li + (j^sw)*G)*8 .. +8, as 4 float pairs
// (pair t: slot t/4, dims 2*(t%4), 2*(t%4)+1 of the chunk).  With two chunks
// per lane the NeoX RoPE partner (i, i + HD/2) of every dim is in the same
// lane.  sw (0/1) swaps the slots of odd groups when a quarter-warp holds two
// groups (G = 4), so its 8 lanes cover all 32 shared-memory banks per load.
template <int HD, int DPL>
struct LaneLayout {
  static constexpr int NCH = DPL / 8;
  static constexpr int G = HD / DPL;
  static constexpr int NP = DPL / 2;
  static constexpr bool kSwap = NCH == 2 && G < 8;
  static __device__ __forceinline__ int chunk_off(int li, int j, int sw) {
    return (li + (j ^ sw) * G) * 8;
  }
  static __device__ __forceinline__ int dim(int li, int t, int sw) {
    return chunk_off(li, t / 4, sw) + 2 * (t % 4);
  }
};

// Load one head vector (fp32) into the lane layout.
template <int HD, int DPL>
__device__ __forceinline__ void load_head_f32(const float* __restrict__ src, int li, int sw,
                                              float2* x) {
  using LL = LaneLayout<HD, DPL>;
#pragma unroll
  for (int j = 0; j < LL::NCH; ++j) {
    const float* p = src + LL::chunk_off(li, j, sw);
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    x[4 * j + 0] = make_float2(a.x, a.y);
    x[4 * j + 1] = make_float2(a.z, a.w);
    x[4 * j + 2] = make_float2(b.x, b.y);
    x[4 * j + 3] = make_float2(b.z, b.w);
  }
}

// Per-head RMSNorm (weight * x * rsqrt(mean(x^2) + eps)) then NeoX RoPE, in
// place, on a head vector in the lane layout.  rope: cos[HD/2], sin[HD/2].
// Warp-uniform (it shuffles).
template <int HD, int DPL>
__device__ __forceinline__ void norm_rope(float2* x, const float* __restrict__ w, float eps,
                                          const float* rope, int li, int sw) {
  using LL = LaneLayout<HD, DPL>;
  constexpr int NP = LL::NP, G = LL::G;
  float ss = 0.f;
#pragma unroll
  for (int t = 0; t < NP; ++t) ss = fmaf(x[t].y, x[t].y, fmaf(x[t].x, x[t].x, ss));
  ss = group_sum<G>(ss);
  const float rinv = 1.0f / sqrtf(ss / (float)HD + eps);
  float2 xn[NP];
#pragma unroll
  for (int t = 0; t < NP; ++t) {
    const int d0 = LL::dim(li, t, sw);
    xn[t] = make_float2(w[d0] * (x[t].x * rinv), w[d0 + 1] * (x[t].y * rinv));
  }
  if constexpr (LL::NCH == 2) {
    // chunk li holds dims i < HD/2 (slot sw), chunk li + G their partners
    // i + HD/2 (slot 1 - sw)
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const int i0 = li * 8 + 2 * p;
      const float c0 = rope[i0], s0 = rope[HD / 2 + i0];
      const float c1 = rope[i0 + 1], s1 = rope[HD / 2 + i0 + 1];
      const float2 lo = sw ? xn[4 + p] : xn[p], hi = sw ? xn[p] : xn[4 + p];
      const float2 ylo = make_float2(lo.x * c0 - hi.x * s0, lo.y * c1 - hi.y * s1);
      const float2 yhi = make_float2(hi.x * c0 + lo.x * s0, hi.y * c1 + lo.y * s1);
      x[p] = sw ? yhi : ylo;
      x[4 + p] = sw ? ylo : yhi;
    }
  } else {
    // one chunk per lane: the partner chunk lives in lane li ^ (G/2)
    const bool lower = li < G / 2;
    const int ib = (lower ? li : li - G / 2) * 8;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float px = __shfl_xor_sync(kFull, xn[p].x, G / 2);
      const float py = __shfl_xor_sync(kFull, xn[p].y, G / 2);
      const int i0 = ib + 2 * p;
      const float c0 = rope[i0], s0 = rope[HD / 2 + i0];
      const float c1 = rope[i0 + 1], s1 = rope[HD / 2 + i0 + 1];
      x[p] = lower ? make_float2(xn[p].x * c0 - px * s0, xn[p].y * c1 - py * s1)
                   : make_float2(xn[p].x * c0 + px * s0, xn[p].y * c1 + py * s1);
    }
  }
}

// cos/sin of p * theta_i for i < HD/2 into rope[] (consumer threads
// 0 .. HD/2-1).  The angle is handled in turns: theta_i / (2 pi) is given as
// an unevaluated float pair (hi + lo, 48 bits).  p * hi is split exactly into
// its rounded value and its error (fmaf), the nearest integer count of turns
// is removed from the rounded part exactly, and the small terms are added
// back, so the fraction f of a turn carries about 2^-24 absolute error for
// any p < 2^24; sincospif then evaluates sin/cos(pi * 2f) with its own
// trivial reduction.
template <int HD>
__device__ __forceinline__ void rope_table(float* rope, const float* turns, int p, int tid) {
  if (tid < HD / 2) {
    const float hi = turns[2 * tid], lo = turns[2 * tid + 1];
    const float pf = (float)p;  // exact for p < 2^24
    const float prod = pf * hi;
    const float err = fmaf(pf, hi, -prod);  // p * hi - prod, exactly
    const float f = (prod - rintf(prod)) + fmaf(pf, lo, err);
    float s, c;
    sincospif(2.0f * f, &s, &c);
    rope[tid] = c;
    rope[HD / 2 + tid] = s;
  }
}

// Row-slot states to shared memory: entry (slot r, virtual head hv, query
// qi) at merge + ((r * Hv + hv) * NQ + qi) * (HD + 4) holds the unnormalised
// output in dimension order, then (max, sum).  Query slots past nq are not
// written (combine_slots skips them).
template <int HD, int NQ, int DPL>
__device__ __forceinline__ void slot_states_out(const float (&M)[NQ], const float (&Ls)[NQ],
                                                const float2 (&O)[NQ][DPL / 2], float* merge,
                                                int r, int hv, int Hv, int li, int sw, int nq) {
  using LL = LaneLayout<HD, DPL>;
#pragma unroll
  for (int qi = 0; qi < NQ; ++qi) {
    if (qi < nq) {
      float* mb = merge + ((r * Hv + hv) * NQ + qi) * (HD + 4);
#pragma unroll
      for (int j = 0; j < LL::NCH; ++j) {
        float4* dst = reinterpret_cast<float4*>(mb + LL::chunk_off(li, j, sw));
        dst[0] = make_float4(O[qi][4 * j].x, O[qi][4 * j].y, O[qi][4 * j + 1].x, O[qi][4 * j + 1].y);
        dst[1] = make_float4(O[qi][4 * j + 2].x, O[qi][4 * j + 2].y, O[qi][4 * j + 3].x,
                             O[qi][4 * j + 3].y);
      }
      if (li == 0) *reinterpret_cast<float2*>(mb + HD) = make_float2(M[qi], Ls[qi]);
    }
  }
}

// Combine the R row-slot states of a CTA's piece of one unit (written by
// slot_states_out) in one pass: each consumer thread takes a slice of 4 * V4
// dimensions of one query, rescales every slot to the common maximum and
// sums.  slot < 0: the unit lies entirely in this CTA and the slice is
// written normalised to the output; else it is written, unnormalised with
// its (max, sum), as partial `slot` of the unit.  members: the source's
// sequences (cross: beams of the group), first at mbase; hg: the unit's
// head group.  V4 = 2 when slices of 4 would outnumber the threads.
template <int HD, int NQ, int V4>
__device__ __forceinline__ void combine_slots(const DecodeArgs& a, const float* merge, int R,
                                              int Hv, int members, int mbase, int hg,
                                              int64_t slot, int tid, int n_cons) {
  constexpr int US = HD / (4 * V4);
  const int hs = a.hs, rep = a.rep;
  const int hqu = hs * rep;  // query heads of a unit
  const int qw = a.Hq * HD;
  const int n = Hv * NQ * US;
  for (int x = tid; x < n; x += n_cons) {
    const int d0 = (x % US) * 4 * V4;
    const int e = x / US;  // entry hv * NQ + qi
    const int qi = e % NQ, hv = e / NQ;
    const int ms = Hv == hs ? 0 : hv / hs, hl = hv - ms * hs;  // no query split: no division
    const int qg = ms * NQ + qi;  // query of the unit's source: member * rep + head offset
    if (qg >= members * rep) continue;  // a query slot past nq: never written
    const float* base = merge + e * (HD + 4);
    const int stride = Hv * NQ * (HD + 4);  // from one row slot's entry to the next
    float M = -INFINITY;
#pragma unroll 4
    for (int r = 0; r < R; ++r) M = fmaxf(M, base[r * stride + HD]);
    float L = 0.f;
    float2 acc[2 * V4];
#pragma unroll
    for (int w = 0; w < 2 * V4; ++w) acc[w] = make_float2(0.f, 0.f);
    if (M != -INFINITY) {
#pragma unroll 4
      for (int r = 0; r < R; ++r) {
        const float* mb = base + r * stride;
        const float2 ml = *reinterpret_cast<const float2*>(mb + HD);
        const float c = ex2(ml.x - M);  // 0 for a slot that saw no rows
        const float2 c2 = make_float2(c, c);
        L = fmaf(ml.y, c, L);
#pragma unroll
        for (int w = 0; w < V4; ++w) {
          const float4 v = *reinterpret_cast<const float4*>(mb + d0 + 4 * w);
          acc[2 * w] = ffma2(c2, make_float2(v.x, v.y), acc[2 * w]);
          acc[2 * w + 1] = ffma2(c2, make_float2(v.z, v.w), acc[2 * w + 1]);
        }
      }
    }
    const int mem = rep == 1 ? qg : qg / rep;
    const int xq = hl * rep + (qg - mem * rep);  // query head within the unit
    if (slot < 0) {
      const float inv = 1.0f / L;
      float* dst = a.out + (int64_t)(mbase + mem) * qw + (hg * hqu + xq) * HD + d0;
#pragma unroll
      for (int w = 0; w < V4; ++w)
        *reinterpret_cast<float4*>(dst + 4 * w) =
            make_float4(acc[2 * w].x * inv, acc[2 * w].y * inv, acc[2 * w + 1].x * inv,
                        acc[2 * w + 1].y * inv);
    } else {
      const int64_t pidx = (slot * a.max_members + mem) * hqu + xq;
#pragma unroll
      for (int w = 0; w < V4; ++w)
        *reinterpret_cast<float4*>(a.part_o + pidx * HD + d0 + 4 * w) =
            make_float4(acc[2 * w].x, acc[2 * w].y, acc[2 * w + 1].x, acc[2 * w + 1].y);
      if (d0 == 0) *reinterpret_cast<float2*>(a.part_ml + pidx * 2) = make_float2(M, L);
    }
  }
}

// The last CTA to finish unit u (source g, head group hg) merges the
// partials of every piece of it (its own among them): each consumer thread
// takes 4 * V4 consecutive output values of one query and combines that
// slice over pieces first..lastp, 8 pieces per L2 round trip, then writes
// it normalised.  The piece of CTA c sits in partial slot c + u.  V4 = 2
// when slices of 4 would outnumber the threads (beam groups: many queries
// per unit), so that each thread makes one pass.
template <int HD, int V4>
__device__ __forceinline__ void merge_pieces(const DecodeArgs& a, int u, int hg, int first,
                                             int lastp, int members, int mbase, int tid,
                                             int n_cons) {
  constexpr int US = HD / (4 * V4);  // slices per head vector
  constexpr int KB = 8;
  const int hqu = a.hs * a.rep;  // query heads of a unit
  const int qw = a.Hq * HD;
  const int nunits = members * hqu * US;
  for (int x = tid; x < nunits; x += n_cons) {
    const int d0 = (x % US) * 4 * V4;
    const int mj = x / US;  // member * hqu + query head within the unit
    const int mem = mj / hqu, j = mj - mem * hqu;
    float M = -INFINITY, Lsum = 0.f;
    float2 acc[2 * V4];
#pragma unroll
    for (int w = 0; w < 2 * V4; ++w) acc[w] = make_float2(0.f, 0.f);
    for (int kb = first; kb <= lastp; kb += KB) {
      float2 ml[KB];
      float4 xv[KB][V4];
#pragma unroll
      for (int i = 0; i < KB; ++i) {
        if (kb + i <= lastp) {
          const int64_t pidx = ((int64_t)(kb + i + u) * a.max_members + mem) * hqu + j;
          ml[i] = __ldcg(reinterpret_cast<const float2*>(a.part_ml + pidx * 2));
#pragma unroll
          for (int w = 0; w < V4; ++w) xv[i][w] = ld_cg_f4(a.part_o + pidx * HD + d0 + 4 * w);
        } else {
          ml[i] = make_float2(-INFINITY, 0.f);
#pragma unroll
          for (int w = 0; w < V4; ++w) xv[i][w] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      float mb = M;
#pragma unroll
      for (int i = 0; i < KB; ++i) mb = fmaxf(mb, ml[i].x);
      if (mb == -INFINITY) continue;
      const float ca = ex2(M - mb);
      const float2 ca2 = make_float2(ca, ca);
      Lsum *= ca;
#pragma unroll
      for (int w = 0; w < 2 * V4; ++w) acc[w] = fmul2(acc[w], ca2);
#pragma unroll
      for (int i = 0; i < KB; ++i) {
        const float c = ex2(ml[i].x - mb);  // 0 for an absent piece
        const float2 c2 = make_float2(c, c);
        Lsum = fmaf(ml[i].y, c, Lsum);
#pragma unroll
        for (int w = 0; w < V4; ++w) {
          acc[2 * w] = ffma2(c2, make_float2(xv[i][w].x, xv[i][w].y), acc[2 * w]);
          acc[2 * w + 1] = ffma2(c2, make_float2(xv[i][w].z, xv[i][w].w), acc[2 * w + 1]);
        }
      }
      M = mb;
    }
    const float inv = 1.0f / Lsum;
    float* dst = a.out + (int64_t)(mbase + mem) * qw + (hg * hqu + j) * HD + d0;
#pragma unroll
    for (int w = 0; w < V4; ++w)
      *reinterpret_cast<float4*>(dst + 4 * w) =
          make_float4(acc[2 * w].x * inv, acc[2 * w].y * inv, acc[2 * w + 1].x * inv,
                      acc[2 * w + 1].y * inv);
  }
}

template <int HD, int NQ, int DPL, int RS, int MAXT>
__global__ void __launch_bounds__(MAXT, 1) decode_attn_kernel(const __grid_constant__ DecodeArgs a) {
  using LL = LaneLayout<HD, DPL>;
  constexpr int G = LL::G, NP = LL::NP, NCH = LL::NCH;
  extern __shared__ __align__(128) unsigned char smem[];
  const int hs = a.hs, HS = a.HS;
  const int Hv = a.MS * hs;  // virtual heads of a unit: (query split, KV head of the group)
  const DecodeSmem lay =
      decode_smem_layout(a.stages, a.n_src, a.R, Hv, NQ, HD, a.stage_elems);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.bars);
  uint64_t* empty = full + a.stages;
  // ctl: [0] abort, [1] ticket, [2] unsorted groups, [3] units to merge,
  // [4 .. 4 + kMergeList) those units
  int* ctl = reinterpret_cast<int*>(smem + lay.ctl);
  int* off = reinterpret_cast<int*>(smem + lay.off);
  int* mst = reinterpret_cast<int*>(smem + lay.mstart);
  int* poff_region = reinterpret_cast<int*>(smem + lay.poff);  // the producer's offsets
  int* slen = reinterpret_cast<int*>(smem + lay.slen);         // length entry per source
  float* rope = reinterpret_cast<float*>(smem + lay.rope);
  float* wts = reinterpret_cast<float*>(smem + lay.wts);  // GQA: RMSNorm weights of q, k
  float* merge = reinterpret_cast<float*>(smem + lay.merge);
  uint16_t* stage = reinterpret_cast<uint16_t*>(smem + lay.stage);
  volatile int* abort_flag = ctl;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_cons = a.R * Hv * G;  // a multiple of 32
  const int cons_warps = n_cons >> 5;
  const int S = a.n_src;
  const int qw = a.Hq * HD;
  const int chunk = a.chunk_elems;  // f16 per row chunk in a stage
  const uint32_t chunk_bytes = (uint32_t)chunk * 2u;
  const int hqu = hs * a.rep;  // query heads of a unit

  if (tid == 0) {
    for (int s = 0; s < a.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], cons_warps);
    }
    for (int i = 0; i < 16; ++i) ctl[i] = 0;
    fence_barrier_init();
  }
  // Let the next kernel on the stream launch now: its CTAs take SMs as ours
  // leave and wait (griddepcontrol.wait) for this grid to finish before they
  // read anything an earlier kernel may write.
  grid_launch_dependents();

  // ---- L2 prefetch of the head of this CTA's share, before the wait.  The
  // K/V history of a step was written by earlier steps, so while the
  // previous kernel drains, the producer warp asks L2 for the first pf_bytes
  // of its share.  The lengths (groups) are read here only to place these
  // hints (from L2, bypassing L1); whatever they hold, every address stays
  // inside the K/V buffer, and a prefetch writes nothing and is never seen by
  // a load, so the hint cannot change a result.  Its offsets go to the stage
  // ring, which nothing touches before this warp's first copy.
  //
  // With the caller's promise that the lengths and the history are ready
  // (a.early) the hints are not needed: the producer starts its copies at
  // once, and the consumers wait only before the queries (below).
  if (!a.early && warp == cons_warps && !a.stall && a.pf_bytes > 0 &&
      2 * (S + 1) * 4 <= a.stages * a.stage_elems * 2) {
    int* poff = reinterpret_cast<int*>(stage);
    int* psq = poff + S + 1;  // beam reorder: the sequence each source reads
    const int run = warp_offsets(a, poff, S, lane, true, nullptr, psq);
    if (run > 0) {
      const int pshare = max((int)((run + gridDim.x - 1) / gridDim.x), a.min_share);
      const int pk0 = (int)min((int64_t)blockIdx.x * pshare, (int64_t)run);
      const int pk1 = min(pk0 + pshare, run);
      // the query rows (and the new token's k, v rows) of the sources the
      // share starts: the same hint, so that the first loads after the wait
      // find them in L2 instead of queueing behind everyone's K/V streams
      if (pk0 < pk1) {
        int lo = 0, hi = S;  // the sources holding pk0 and pk1 - 1
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (poff[mid] <= pk0) lo = mid;
          else hi = mid;
        }
        const int g0 = lo;
        hi = S;
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (poff[mid] <= pk1 - 1) lo = mid;
          else hi = mid;
        }
        const int g1 = min(lo, g0 + 63);
        const uint32_t qbytes = (uint32_t)a.Hq * HD * 4;
        if (a.mode == kModeCross) {
          for (int b = lane; b < a.B; b += 32) {
            const int gr = __ldcg(a.group + b);
            if (gr >= g0 && gr <= g1) bulk_prefetch_l2(a.q + (int64_t)b * a.q_stride, qbytes);
          }
        } else {
          for (int g = g0 + lane; g <= g1; g += 32) {
            bulk_prefetch_l2(a.q + (int64_t)g * a.q_stride, qbytes);
            if (a.append) {
              bulk_prefetch_l2(a.k_new + (int64_t)g * a.kv_stride, (uint32_t)a.Hkv * HD * 4);
              bulk_prefetch_l2(a.v_new + (int64_t)g * a.kv_stride, (uint32_t)a.Hkv * HD * 4);
            }
          }
        }
      }
      if (lane == 0 && pk0 < pk1) {
        TileIter it(poff, S, HS, pk0, pk1, a.tile_rows, a.seg_rows);
        Tile tl;
        int left = a.pf_bytes;
        while (left > 0 && it.next(tl)) {
          if (HS == 1) {
            const int sq = a.idx ? psq[tl.g] : tl.g;
            bulk_prefetch_l2(a.kv + (int64_t)sq * a.src_stride + (int64_t)tl.row0 * a.row_elems,
                             (uint32_t)tl.nr * chunk_bytes);
          } else {
            for (int rr = 0; rr < tl.nr; rr += kBoxRows)
              tma_prefetch_5d(&a.tmap_rows, tl.hg * hs, 0, tl.row0 + rr, tl.g);
          }
          left -= tl.nr * (int)chunk_bytes;
        }
      }
    }
    __syncwarp();
  }
  __syncthreads();  // barrier initialisation and ctl are visible to every warp
  if (!a.early) grid_dependency_wait();

  if (warp == cons_warps) {
    // ======================= producer warp: one lane issues the copies.  It
    // computes the offsets itself (the same integers the consumers compute)
    // and starts at once.
    int* toff = poff_region;
    int* tsq = reinterpret_cast<int*>(smem + lay.psrc);
    const int total = warp_offsets(a, toff, S, lane, false, nullptr, tsq);
    if (total <= 0 || a.stall) {  // nothing to stream, unsorted groups, or the stall test
      grid_launch_dependents();
      return;
    }
    const int share = max((int)((total + gridDim.x - 1) / gridDim.x), a.min_share);
    const int k0 = (int)min((int64_t)blockIdx.x * share, (int64_t)total);
    const int k1 = min(k0 + share, total);
    if (lane == 0 && k0 < k1) {
      const uint64_t pol = policy_evict_first();
      // Beam reorder (whole rows, HS == 1): each tile, once it has landed, is
      // also stored to its destination sequence.  The stores trail the loads
      // by stages - 1 tiles (a second walker `st` names them), so waiting for
      // the tile to store never holds back a load the ring has room for; the
      // store of the tile a stage held has read it before the stage is
      // loaded again.
      const bool reorder = a.idx != nullptr;
      TileIter it(toff, S, HS, k0, k1, a.tile_rows, a.seg_rows);
      TileIter st(toff, S, HS, k0, k1, a.tile_rows, a.seg_rows);
      Tile tl, ts;
      int t = 0, stored = 0;
      bool aborted = false;
      auto store_next = [&]() -> bool {
        const int j = stored;
        if (!st.next(ts) || !mbar_wait(&full[j % a.stages], (j / a.stages) & 1, a.wait_ns))
          return false;
        bulk_s2g(a.cache_w + (int64_t)ts.g * a.src_stride + (int64_t)ts.row0 * a.row_elems,
                 stage + (size_t)(j % a.stages) * a.stage_elems, (uint32_t)ts.nr * chunk_bytes);
        bulk_commit();
        ++stored;
        return true;
      };
      for (; it.next(tl); ++t) {
        const int s = t % a.stages;
        if (t >= a.stages && !mbar_wait(&empty[s], ((t / a.stages) - 1) & 1, a.wait_ns)) {
          aborted = true;
          break;
        }
        if (*abort_flag) break;  // the consumers gave up: issue nothing more
        if (reorder && t >= a.stages) bulk_wait_read();  // tile t - stages is stored
        uint16_t* dst = stage + (size_t)s * a.stage_elems;
        mbar_arrive_expect_tx(&full[s], (uint32_t)tl.nr * chunk_bytes);
        if (HS == 1) {
          const int sq = reorder ? tsq[tl.g] : tl.g;
          bulk_g2s(dst, a.kv + (int64_t)sq * a.src_stride + (int64_t)tl.row0 * a.row_elems,
                   (uint32_t)tl.nr * chunk_bytes, &full[s], pol);
          if (reorder && t >= a.stages - 1 && !store_next()) {
            ++t;  // tile t was issued: the drain below covers it
            aborted = true;
            break;
          }
        } else {
          const int c1 = tl.hg * hs;
          int rr = 0;
          for (; rr + kBoxRows <= tl.nr; rr += kBoxRows)
            tma_load_5d(dst + (size_t)rr * chunk, &a.tmap_rows, c1, 0, tl.row0 + rr, tl.g, &full[s],
                        pol);
          for (; rr < tl.nr; ++rr)
            tma_load_5d(dst + (size_t)rr * chunk, &a.tmap_row, c1, 0, tl.row0 + rr, tl.g, &full[s],
                        pol);
        }
      }
      // the tiles still to store
      if (reorder && !aborted && *abort_flag == 0) {
        while (stored < t) {
          if (!store_next()) {
            aborted = true;
            break;
          }
        }
      }
      if (aborted) {
        set_dev_err(a.dev_err, ASR_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      // The CTA must not end while a copy into or out of its shared memory
      // is in flight: wait (bounded) until the last loads issued have landed,
      // then for the stores (which read only landed tiles and always finish).
      for (int t2 = max(0, t - a.stages); t2 < t; ++t2)
        if (!mbar_wait(&full[t2 % a.stages], (t2 / a.stages) & 1, a.wait_ns))
          set_dev_err(a.dev_err, ASR_DEVERR_TIMEOUT);
      if (reorder) bulk_wait_all();
    }
    grid_launch_dependents();
    return;
  }
  if (warp > cons_warps) return;

  // ---- consumers: keys per source (off) and first sequence per source (mst)
  if (a.mode != kModeCross) {
    // Self / GQA: one warp computes the offsets (the other warps load the
    // RMSNorm weights meanwhile); one sequence per source, so mst[g] = g.
    if (warp == 0) {
      warp_offsets(a, off, S, lane, false, slen);
      for (int g = lane; g <= S; g += 32) mst[g] = g;
    }
    if (a.mode == kModeGqa) {
      const int t0 = n_cons > 32 ? 32 : 0;
      if (tid >= t0)
        for (int i = tid - t0; i < 2 * HD; i += n_cons - t0) wts[i] = i < HD ? a.wq[i] : a.wk[i - HD];
    }
  } else {
    // Cross: warp 0 computes the offsets, the other warps the first
    // sequence of each group.
    if (warp == 0) {
      if (warp_offsets(a, off, S, lane, false) < 0 && lane == 0) ctl[2] = 1;
    } else {
      first_members(a, mst, S, tid - 32, n_cons - 32);
    }
  }
  named_bar(1, n_cons);
  // the queries, the new token, the outputs and the workspace belong to
  // earlier grids: with the caller's promise, the wait comes only now
  if (a.early) grid_dependency_wait();
  const bool unsorted = a.mode == kModeCross && ctl[2] != 0;

  // ---- CTA 0 zeroes the outputs of sequences that are skipped
  if (blockIdx.x == 0) {
    for (int b = warp; b < a.B; b += cons_warps) {
      int bad = 0;
      if (unsorted) {
        bad = ASR_DEVERR_INDEX;
      } else if (a.mode == kModeCross) {
        const int gr = a.group[b];
        if (gr < 0 || gr >= S) bad = ASR_DEVERR_INDEX;
        else if (b - mst[gr] >= a.max_members) bad = ASR_DEVERR_BEAMS;
      } else {
        const int v = slen[b];
        const bool ok =
            a.mode == kModeSelf ? (v >= 1 && v <= a.capacity) : (v >= 0 && v < a.capacity);
        if (!ok) bad = (a.idx && (unsigned)a.idx[b] >= (unsigned)S) ? ASR_DEVERR_INDEX : ASR_DEVERR_LEN;
        if (a.lens_out && lane == 0) a.lens_out[b] = bad ? 0 : v;
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

  // ---- this CTA's share of the flattened key axis (the producer's too)
  const int total = off[S];
  const int P = gridDim.x;
  const int share = max((total + P - 1) / P, a.min_share);
  const int k0 = (int)min((int64_t)blockIdx.x * share, (int64_t)total);
  const int k1 = min(k0 + share, total);

  // ======================= consumers
  // group grp: virtual head hv = (query split ms, KV head hl of the unit's
  // group), row slot r
  const int grp = tid / G, li = tid % G;
  const int hv = grp % Hv, r = grp / Hv;
  const int hl = hv % hs, ms = hv / hs;
  const int qb = ms * NQ;  // this group's first query of a source
  const int rep = a.rep;
  const int R = a.R;
  const int sw = LL::kSwap ? (grp & 1) : 0;
  const int hoff = hl * HD;  // element offset of this group's head in a chunk's K (or V) half
  const int voff = hs * HD;  // element offset of the V half of a chunk

  float2 qv[NQ][NP], o[NQ][NP];
  float m[NQ], l[NQ];
  int nq = 0, mbase = 0, h = 0;

  // Append: the new token's key/value (GQA: normed and roped) from kx, vx
  // (fp32, loaded by the caller), written to the cache by row slot 0 as f16,
  // then folded, with the value the cache holds, into the running state of
  // row slot 0 as the first key it sees.  Warp-uniform (it may shuffle).
  auto append_fold = [&](int g, float2* kx, float2* vx) {
    const int p = a.mode == kModeGqa ? slen[g] : slen[g] - 1;
    if (a.mode == kModeGqa) norm_rope<HD, DPL>(kx, wts + HD, a.eps, rope, li, sw);
    uint16_t* row = a.cache_w + (int64_t)g * a.src_stride + (int64_t)p * a.row_elems;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      float kf[8], vf[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        kf[2 * e] = kx[4 * j + e].x;
        kf[2 * e + 1] = kx[4 * j + e].y;
        vf[2 * e] = vx[4 * j + e].x;
        vf[2 * e + 1] = vx[4 * j + e].y;
      }
      const uint4 kh = f8_to_h8(kf), vh = f8_to_h8(vf);
      h8_to_f2x4(kh, kx + 4 * j);  // the key and value as the cache holds them
      h8_to_f2x4(vh, vx + 4 * j);
      if (r == 0 && ms == 0) {
        *reinterpret_cast<uint4*>(row + h * HD + LL::chunk_off(li, j, sw)) = kh;
        *reinterpret_cast<uint4*>(row + a.Hkv * HD + h * HD + LL::chunk_off(li, j, sw)) = vh;
      }
    }
    // every query slot runs the group sum (its shuffles need the whole warp,
    // and groups of one warp may hold different query counts); slots past
    // nq hold zero queries and are not kept
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) {
      {
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int t = 0; t < NP; ++t) acc = ffma2(qv[qi][t], kx[t], acc);
        const float sc = group_sum<G>(acc.x + acc.y);
        if (r == 0 && qi < nq) {  // one row slot holds it; the slots are merged later
          m[qi] = sc;  // exp2(score - m) = 1
          l[qi] = 1.f;
#pragma unroll
          for (int t = 0; t < NP; ++t) o[qi][t] = vx[t];
        }
      }
    }
  };

  // Start unit u: its queries, and the new token in the CTA that folds it
  // in.  Warp-uniform.
  auto seg_begin = [&](int u) {
    const int g = u / HS, hg = u - g * HS;
    h = hg * hs + hl;  // this group's KV head
    mbase = mst[g];
    nq = min(max(min(mst[g + 1] - mst[g], a.max_members) * rep - qb, 0), NQ);
    const bool fold = a.append && owns_first_row(off, HS, a.seg_rows, share, u, (int)blockIdx.x);
    // member m, query head x of the unit at qsrc + m * q_stride + x * HD;
    // every global load (new token, queries) is issued before the RoPE
    // table is built, so their latencies overlap it and one another
    const float* qsrc = a.q + (int64_t)mbase * a.q_stride + (int64_t)hg * hqu * HD;
    const float* ksrc = a.k_new + (int64_t)g * a.kv_stride + h * HD;
    const float* vsrc = a.v_new + (int64_t)g * a.kv_stride + h * HD;
    float2 kx[NP], vx[NP];
    if (fold) {
      load_head_f32<HD, DPL>(ksrc, li, sw, kx);
      load_head_f32<HD, DPL>(vsrc, li, sw, vx);
    }
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) {
      m[qi] = -INFINITY;
      l[qi] = 0.f;
#pragma unroll
      for (int t = 0; t < NP; ++t) o[qi][t] = make_float2(0.f, 0.f);
      if (qi < nq) {
        const int mem = (qb + qi) / rep;
        const int x = hl * rep + (qb + qi) % rep;  // query head within the unit
        load_head_f32<HD, DPL>(qsrc + mem * a.q_stride + x * HD, li, sw, qv[qi]);
      } else {
#pragma unroll
        for (int t = 0; t < NP; ++t) qv[qi][t] = make_float2(0.f, 0.f);
      }
    }
    if (a.mode == kModeGqa) {
      named_bar(1, n_cons);
      rope_table<HD>(rope, a.rope_turns, slen[g], tid);
      named_bar(1, n_cons);
    }
    const float2 s2 = make_float2(a.qscale, a.qscale);
    // warp-uniform: norm_rope shuffles (slots past nq hold zeros)
#pragma unroll
    for (int qi = 0; qi < NQ; ++qi) {
      if (a.mode == kModeGqa) norm_rope<HD, DPL>(qv[qi], wts, a.eps, rope, li, sw);
#pragma unroll
      for (int t = 0; t < NP; ++t) qv[qi][t] = fmul2(qv[qi][t], s2);
    }
    if (fold) append_fold(g, kx, vx);
  };

  // The merge of unit u's partials by the last CTA to finish it.
  auto merge_unit = [&](int u) {
    const UnitSpan sp = unit_span(off, HS, a.seg_rows, u);
    const int first = sp.go / share, lastp = (sp.go + sp.gl - 1) / share;
    const int g = u / HS;
    const int members = min(mst[g + 1] - mst[g], a.max_members);
    // wider slices only where several queries share a unit (one query per
    // KV head always has a thread per slice)
    if (NQ > 1 && members * hs * rep * (HD / 4) > n_cons)
      merge_pieces<HD, (NQ > 1 ? 2 : 1)>(a, u, u - g * HS, first, lastp, members, mst[g], tid,
                                         n_cons);
    else
      merge_pieces<HD, 1>(a, u, u - g * HS, first, lastp, members, mst[g], tid, n_cons);
  };

  // The end of this CTA's piece of unit u: the row slots' states meet in
  // shared memory and are combined slice by slice (one barrier pair, no
  // tree), straight into the output when the CTA holds the whole unit, else
  // into this piece's partial, which the last CTA to finish the unit merges.
  auto seg_end = [&](int u) {
    named_bar(1, n_cons);  // the previous readers of the buffer are done
    slot_states_out<HD, NQ, DPL>(m, l, o, merge, r, hv, Hv, li, sw, nq);
    named_bar(1, n_cons);
    // pieces of this unit over the grid
    const UnitSpan sp = unit_span(off, HS, a.seg_rows, u);
    const int first = sp.gl > 0 ? sp.go / share : 0;
    const int lastp = sp.gl > 0 ? (sp.go + sp.gl - 1) / share : 0;
    const int parts = sp.gl > 0 ? lastp - first + 1 : 0;
    const int g = u / HS;
    const int64_t pslot = parts > 1 ? (int64_t)blockIdx.x + u : -1;
    const int members = min(mst[g + 1] - mst[g], a.max_members);
    if (NQ > 1 && Hv * NQ * (HD / 4) > n_cons)
      combine_slots<HD, NQ, (NQ > 1 ? 2 : 1)>(a, merge, R, Hv, members, mst[g], u - g * HS, pslot,
                                              tid, n_cons);
    else
      combine_slots<HD, NQ, 1>(a, merge, R, Hv, members, mst[g], u - g * HS, pslot, tid, n_cons);
    if (parts <= 1) return;
    // ticket: the barrier orders the CTA's partial writes before thread 0's
    // release; the acquire side lets the last CTA read everyone's partials
    named_bar(1, n_cons);
    if (tid == 0) {
      const int old = atomic_add_acq_rel_gpu(&a.counters[u], 1);
      const int is_last = old == parts - 1;
      if (is_last) a.counters[u] = 0;  // no other CTA touches it again in this launch
      ctl[1] = is_last;
    }
    named_bar(1, n_cons);
    if (ctl[1]) {
      // the last CTA to finish unit u merges every piece's partial, after
      // its tiles (the last arrival is nearly always at the end of a share
      // anyway, and outside the tile loop the merge has the registers)
      named_bar(1, n_cons);  // every thread has read ctl[1]
      if (tid == 0) ctl[4 + ctl[3]++] = u;
    }
  };

  if (k0 < k1) {
    TileIter it(off, S, HS, k0, k1, a.tile_rows, a.seg_rows);
    Tile tl;
    for (int t = 0; it.next(tl); ++t) {
      if (tl.first) seg_begin(tl.u);
      const int s = t % a.stages;
      // A wait that runs out aborts the CTA: every warp then passes over its
      // remaining tiles without waiting or reading them (so the control flow,
      // named barriers and tickets stay the same in every warp) and the
      // producer issues nothing more.  The outputs of such a call are
      // undefined; ASR_DEVERR_TIMEOUT tells the host.
      bool ok = __shfl_sync(kFull, *abort_flag, 0) == 0;
      if (ok) ok = __all_sync(kFull, mbar_wait(&full[s], (t / a.stages) & 1, a.wait_ns));
      if (!ok && lane == 0 && *abort_flag == 0) {
        *abort_flag = 1;
        set_dev_err(a.dev_err, ASR_DEVERR_TIMEOUT);
      }
      if (ok) {
        const uint16_t* tb = stage + (size_t)s * a.stage_elems + hoff;
        // scores of this group's rows (row r + i*R of the tile)
        float sc[NQ][RS];
        bool val[RS];
#pragma unroll
        for (int i = 0; i < RS; ++i) {
          const int row = r + i * R;  // < tile_rows: always inside the stage buffer
          val[i] = row < tl.nr;
          float2 kf[NP];
#pragma unroll
          for (int j = 0; j < NCH; ++j) {
            const uint4 uu = *reinterpret_cast<const uint4*>(tb + row * chunk + LL::chunk_off(li, j, sw));
            h8_to_f2x4(uu, kf + 4 * j);
          }
          // every query slot is scored and reduced: the reduction's
          // shuffles need the whole warp, and the groups of one warp may hold
          // different query counts (slots past nq hold zero queries)
#pragma unroll
          for (int qi = 0; qi < NQ; ++qi) {
            float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
            for (int t2 = 0; t2 < NP; t2 += 2) {
              a0 = ffma2(qv[qi][t2], kf[t2], a0);
              a1 = ffma2(qv[qi][t2 + 1], kf[t2 + 1], a1);
            }
            sc[qi][i] = (a0.x + a0.y) + (a1.x + a1.y);
          }
        }
#pragma unroll
        for (int o2 = 1; o2 < G; o2 <<= 1) {
#pragma unroll
          for (int qi = 0; qi < NQ; ++qi) {
#pragma unroll
            for (int i = 0; i < RS; ++i) sc[qi][i] += __shfl_xor_sync(kFull, sc[qi][i], o2);
          }
        }
        // online softmax over the RS rows, one rescale per tile.  Every query
        // slot runs it (no branch on nq in the loop); a slot past nq holds a
        // zero query, stays finite and is never written out.
        float pr[NQ][RS];
#pragma unroll
        for (int qi = 0; qi < NQ; ++qi) {
#pragma unroll
          for (int i = 0; i < RS; ++i) pr[qi][i] = 0.f;
          {
            float mt = -INFINITY;
#pragma unroll
            for (int i = 0; i < RS; ++i)
              if (val[i]) mt = fmaxf(mt, sc[qi][i]);
            if (mt != -INFINITY) {
              const float mn = fmaxf(m[qi], mt);
              const float alpha = ex2(m[qi] - mn);
              float psum = 0.f;
#pragma unroll
              for (int i = 0; i < RS; ++i) {
                pr[qi][i] = val[i] ? ex2(sc[qi][i] - mn) : 0.f;
                psum += pr[qi][i];
              }
              l[qi] = fmaf(l[qi], alpha, psum);
              m[qi] = mn;
              const float2 al2 = make_float2(alpha, alpha);
#pragma unroll
              for (int t2 = 0; t2 < NP; ++t2) o[qi][t2] = fmul2(o[qi][t2], al2);
            }
          }
        }
        // weighted values
#pragma unroll
        for (int i = 0; i < RS; ++i) {
          if (val[i]) {
            const int row = r + i * R;
            float2 vf[NP];
#pragma unroll
            for (int j = 0; j < NCH; ++j) {
              const uint4 uu = *reinterpret_cast<const uint4*>(tb + row * chunk + voff +
                                                               LL::chunk_off(li, j, sw));
              h8_to_f2x4(uu, vf + 4 * j);
            }
#pragma unroll
            for (int qi = 0; qi < NQ; ++qi) {
              const float2 p2 = make_float2(pr[qi][i], pr[qi][i]);
#pragma unroll
              for (int t2 = 0; t2 < NP; ++t2) o[qi][t2] = ffma2(p2, vf[t2], o[qi][t2]);
            }
          }
        }
      }
      // the stage is consumed (or abandoned): hand it back to the producer
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (tl.last) seg_end(tl.u);
    }
  }

  // Appending units with no cached rows (GQA n_past == 0, self lens == 1):
  // only the new token; CTA u % P handles unit u.
  if (a.append) {
    for (int u = blockIdx.x; u < a.n_units; u += P) {
      if (slen[u / HS] == (a.mode == kModeGqa ? 0 : 1)) {
        seg_begin(u);
        seg_end(u);
      }
    }
  }
  // the merges this CTA won (ctl[3] was last written before a barrier)
  named_bar(1, n_cons);
  for (int i = 0; i < ctl[3]; ++i) merge_unit(ctl[4 + i]);
  grid_launch_dependents();
}

// ---------------------------------------------------------------- host ----

// Per query-count bucket: dims per lane, rows per slot per tile, thread cap.
struct Variant {
  int NQ, DPL, RS, MAXT;
};
static constexpr int kNumVariants = 5;
static constexpr Variant kVariants[kNumVariants] = {
    {1, 16, 4, 384}, {2, 16, 4, 384}, {4, 8, 2, 384}, {8, 8, 2, 256},
    // the GQA step at head_dim 128 with two query heads per KV head: five
    // rows per thread and tile, and at most 256 threads (7 row slots), so a
    // thread may hold 255 registers rather than 168 (the compiler budgets a
    // launch bound's threads in multiples of 128): its consumers bound the
    // tiles, and this measured 2 % faster than four rows in 10 slots, which
    // the beam-group cross launches keep
    {2, 16, 5, 256}};
static constexpr int kGqaVariant = 4;

static int variant_index(int nq) {
  if (nq <= 1) return 0;
  if (nq <= 2) return 1;
  if (nq <= 4) return 2;
  if (nq <= 8) return 3;
  return -1;
}

template <int HD, int VI>
static void* kernel_ptr() {
  constexpr Variant v = kVariants[VI];
  return (void*)decode_attn_kernel<HD, v.NQ, v.DPL, v.RS, v.MAXT>;
}

static void* kernel_for(int HD, int vi) {
  if (HD == 64) {
    switch (vi) {
      case 0: return kernel_ptr<64, 0>();
      case 1: return kernel_ptr<64, 1>();
      case 2: return kernel_ptr<64, 2>();
      case 3: return kernel_ptr<64, 3>();
    }
  } else if (HD == 128) {
    switch (vi) {
      case 0: return kernel_ptr<128, 0>();
      case 1: return kernel_ptr<128, 1>();
      case 2: return kernel_ptr<128, 2>();
      case 3: return kernel_ptr<128, 3>();
      case kGqaVariant: return kernel_ptr<128, kGqaVariant>();
    }
  }
  return nullptr;
}

// Tuning constants (measured on GB300): one CTA per SM with about ten
// consumer warps and two or more stages of large tiles.
//   tile_kb: largest K/V tile (bytes of row chunks) one stage holds;
//   smem_kb: shared memory the stage ring may fill;
//   min_kb: fewest K/V bytes one CTA takes (bounds the partials per unit);
//   seg_kb: K/V bytes' worth of virtual rows charged to each unit, so CTAs
//     that start or finish more units take fewer rows (gqa_seg_kb for the
//     GQA step, whose unit start also normalises and rotates its queries);
//   qs: queries per thread group when a KV row serves more than two queries;
//   parts: the number of CTA pieces per unit the head split aims at (a
//     source is cut into the fewest head groups that bring its expected
//     pieces to this or below);
//   min_chunk: fewest bytes of one row a head group streams.
struct DecodeTune {
  int tile_kb = 80, smem_kb = 200, min_kb = 64, seg_kb = 256, gqa_seg_kb = 384, qs = 2, parts = 6,
      min_chunk = 512;
};

static constexpr DecodeTune decode_tune() { return DecodeTune{}; }

struct DecodePlan {
  int vi, MS, HS, hs, R, tile_rows, stages, stage_elems, threads, smem, min_share, seg_rows,
      pf_bytes;
};

// Row slots R: the consumer count R * Hv * G must be a multiple of 32 and
// fit the variant's thread cap (at most 320 consumers), and two stages plus
// the slots' merge entries must fit in shared memory; among those, the
// largest R whose tile fits tile_kb (else the smallest valid R).  Stages: as
// many as fit smem_kb, 2..8.  One CTA takes at least min_kb of rows, so a
// unit splits into a bounded number of partial results.
static bool plan_layout(const DecodeArgs& a, int HD, int vi, int MS, int hs, DecodePlan& p) {
  const int seg_kb = a.mode == kModeGqa ? decode_tune().gqa_seg_kb : decode_tune().seg_kb;
  const int n_src = a.n_src;
  const DecodeTune tune = decode_tune();
  const Variant& v = kVariants[vi];
  const int G = HD / v.DPL;
  const int per_slot = MS * hs * G;
  const int budget = std::min(v.MAXT - 32, 320);
  const int chunk_elems = 2 * hs * HD;
  const int chunk_bytes = chunk_elems * 2;
  int best = 0, smallest = 0;
  for (int R = 1; R * per_slot <= budget; ++R) {
    if ((R * per_slot) % 32 != 0) continue;
    // two stages and the R slots' merge entries must fit a CTA's shared memory
    const int se = dsm_align(R * v.RS * chunk_elems, 64);
    if (decode_smem_layout(2, n_src, R, MS * hs, v.NQ, HD, se).total > 227 * 1024) break;
    if (!smallest) smallest = R;
    if (R * v.RS * chunk_bytes <= tune.tile_kb * 1024) best = R;
  }
  if (!best) best = smallest;
  if (!best) return false;
  p.vi = vi;
  p.MS = MS;
  p.hs = hs;
  p.R = best;
  p.threads = best * per_slot + 32;
  p.tile_rows = best * v.RS;
  p.stage_elems = dsm_align(p.tile_rows * chunk_elems, 64);
  const int cap = tune.smem_kb * 1024;
  int stages = 8;
  while (stages > 2 &&
         decode_smem_layout(stages, n_src, p.R, MS * hs, v.NQ, HD, p.stage_elems).total > cap)
    --stages;
  p.stages = stages;
  p.smem = decode_smem_layout(stages, n_src, p.R, MS * hs, v.NQ, HD, p.stage_elems).total;
  if (p.smem > 227 * 1024) return false;
  p.min_share = std::max(p.tile_rows, (tune.min_kb * 1024 + chunk_bytes - 1) / chunk_bytes);
  p.seg_rows = seg_kb * 1024 / chunk_bytes;
  p.pf_bytes = stages * p.tile_rows * chunk_bytes;
  return true;
}

// The variant and query split (more than two queries per KV row, the beams
// of a group, are split over groups of threads, `qs` queries each: fewer
// registers per thread, more warps per SM), then the head split: the fewest
// head groups per source whose expected pieces per unit are at most
// `parts`.  The expectation takes each source at half its capacity (self,
// GQA) or at its frames (cross), spread over one CTA per SM.
static bool plan_decode(const DecodeArgs& a, int HD, int nq_needed, int sms, DecodePlan& p) {
  const DecodeTune tune = decode_tune();
  int MS = 1, nq_var = nq_needed;
  if (tune.qs > 0 && tune.qs < nq_needed) {
    nq_var = tune.qs;
    MS = (nq_needed + tune.qs - 1) / tune.qs;
  }
  int vi = variant_index(nq_var);
  if (vi < 0) return false;
  if (a.mode == kModeGqa && vi == 1 && HD == 128) vi = kGqaVariant;
  const double rows = a.mode == kModeCross ? (double)a.fixed_len : 0.5 * a.capacity;
  const double row_bytes = 2.0 * a.row_elems;
  const double share = std::max(a.n_src * rows * row_bytes / sms, tune.min_kb * 1024.0);
  bool found = false;
  for (int pass = 0; pass < 2 && !found; ++pass) {
    if (pass == 1) {  // the split's thread layout does not fit: one group per KV head
      MS = 1;
      vi = variant_index(nq_needed);
      if (vi < 0) return false;
    }
    // Cross-attention keeps whole rows: its beams already share each row
    // among several queries, and splitting the heads measured slower there.
    // The beam reorder stores whole landed rows, so it keeps them too.
    const int max_hs_split = (a.mode == kModeCross || a.idx) ? 1 : a.Hkv;
    for (int HS = 1; HS <= max_hs_split; ++HS) {
      if (a.Hkv % HS != 0) continue;
      const int hs = a.Hkv / HS;
      if (HS > 1 && 4 * hs * HD < tune.min_chunk) break;
      DecodePlan c;
      if (!plan_layout(a, HD, vi, MS, hs, c)) continue;
      c.HS = HS;
      p = c;
      found = true;
      if (rows * row_bytes / HS / share <= tune.parts) break;
    }
  }
  return found;
}

static size_t counter_bytes(int n_src, int Hq) { return align_up((size_t)n_src * Hq * 4, 256); }

size_t decode_counter_bytes(int n_src, int Hq) { return counter_bytes(n_src, Hq); }

// Partial results: one slot per (CTA piece, unit), each with max_members x
// (query heads of the unit) entries; (P + n_src * HS) * hs * rep <= (P +
// n_src) * Hq for every head split, so one size serves them all.
size_t decode_ws_bytes(int n_src, int max_members, int Hq, int HD, int sms) {
  const int64_t entries = ((int64_t)kMaxCtasPerSm * sms + n_src) * max_members * Hq;
  const size_t ml = align_up((size_t)entries * 2 * 4, 256);
  const size_t o = (size_t)entries * HD * 4;
  return counter_bytes(n_src, Hq) + ml + o;
}

// CTAs per SM for (kernel, threads, smem) on the current device; the query
// is slow next to a launch, so results are memoised (small linear table).
static int occupancy_cached(void* fn, int threads, int smem) {
  struct Entry {
    void* fn;
    int dev, threads, smem, occ;
  };
  static Entry table[64];
  static int n = 0;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (table[i].fn == fn && table[i].dev == dev && table[i].threads == threads &&
        table[i].smem == smem)
      return table[i].occ;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, fn, threads, smem) != cudaSuccess)
    return 0;
  if (n < 64) table[n++] = {fn, dev, threads, smem, occ};
  return occ;
}

// Test support (asr_debug_stall_next_decode): the next decode launch made by
// this host thread issues no copies and bounds its waits by this many ns.
static thread_local uint64_t t_stall_ns = 0;

// asr_set_history_ready: the decode launches of this host thread read the
// lengths and the cached history before the grid dependency wait.
static thread_local int t_history_ready = 0;

static int launch_decode(DecodeArgs& a, int HD, int nq_needed, void* ws, size_t ws_bytes,
                         cudaStream_t stream) {
  const int sms = device_sm_count();
  if (sms <= 0) return ASR_ERR_CUDA;
  DecodePlan p;
  if (!plan_decode(a, HD, nq_needed, sms, p)) return ASR_ERR_UNSUPPORTED;
  const size_t need = decode_ws_bytes(a.n_src, a.max_members, a.Hq, HD, sms);
  if (!ws || ((uintptr_t)ws & 255u) != 0 || ws_bytes < need) return ASR_ERR_WORKSPACE;
  void* fn = kernel_for(HD, p.vi);
  if (ensure_dynamic_smem(fn, 227 * 1024) != cudaSuccess) return ASR_ERR_CUDA;
  int occ = occupancy_cached(fn, p.threads, p.smem);
  if (occ <= 0) return ASR_ERR_CUDA;
  occ = std::max(1, std::min(occ, kMaxCtasPerSm));
  a.MS = p.MS;
  a.HS = p.HS;
  a.hs = p.hs;
  a.chunk_elems = 2 * p.hs * HD;
  a.n_units = a.n_src * p.HS;
  char* w = static_cast<char*>(ws);
  a.counters = reinterpret_cast<int*>(w);
  w += counter_bytes(a.n_src, a.Hq);
  const int64_t entries = ((int64_t)kMaxCtasPerSm * sms + a.n_src) * a.max_members * a.Hq;
  a.part_ml = reinterpret_cast<float*>(w);
  w += align_up((size_t)entries * 2 * 4, 256);
  a.part_o = reinterpret_cast<float*>(w);
  a.R = p.R;
  a.tile_rows = p.tile_rows;
  a.min_share = p.min_share;
  a.seg_rows = p.seg_rows;
  a.stages = p.stages;
  a.pf_bytes = p.pf_bytes;
  a.stage_elems = p.stage_elems;
  a.wait_ns = kWaitLimitNs;
  a.stall = 0;
  if (t_stall_ns) {
    a.wait_ns = t_stall_ns;
    a.stall = 1;
    t_stall_ns = 0;
  }
  // never for a beam reorder (it writes a destination cache) or the stall test
  a.early = t_history_ready && a.idx == nullptr && !a.stall ? 1 : 0;
  if (p.HS > 1) {
    // rows of every source as {HD, Hkv, 2 (K, V), rows, sources}: a box of
    // {HD, hs, 2, n, 1} lands as n row chunks [K of the hs heads | V of them]
    const uint64_t rows = a.mode == kModeCross ? (uint64_t)a.fixed_len : (uint64_t)a.capacity;
    const uint64_t dims[5] = {(uint64_t)HD, (uint64_t)a.Hkv, 2, rows, (uint64_t)a.n_src};
    const uint64_t strides[4] = {(uint64_t)HD * 2, (uint64_t)a.Hkv * HD * 2,
                                 (uint64_t)a.row_elems * 2, (uint64_t)a.src_stride * 2};
    const uint32_t box_rows[5] = {(uint32_t)HD, (uint32_t)p.hs, 2, (uint32_t)kBoxRows, 1};
    const uint32_t box_row[5] = {(uint32_t)HD, (uint32_t)p.hs, 2, 1, 1};
    if (!make_tmap_f16_5d_plain(&a.tmap_rows, a.kv, dims, strides, box_rows) ||
        !make_tmap_f16_5d_plain(&a.tmap_row, a.kv, dims, strides, box_row))
      return ASR_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sms * occ);
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

// The flattened key axis is int: every source's rows plus its virtual rows,
// once per head group, must fit.
static bool rows_fit_int(int64_t n_src, int64_t rows, int64_t kv_heads) {
  return n_src * (rows + 1024) * kv_heads < (1LL << 31);
}

}  // namespace asrkv

using namespace asrkv;

extern "C" int asr_set_history_ready(int ready) {
  if (ready != 0 && ready != 1) return ASR_ERR_INVALID_ARG;
  t_history_ready = ready;
  return ASR_OK;
}

extern "C" int asr_debug_stall_next_decode(uint64_t wait_ns) {
  if (wait_ns == 0 || wait_ns > kWaitLimitNs) return ASR_ERR_INVALID_ARG;
  t_stall_ns = wait_ns;
  return ASR_OK;
}

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
  if (!rows_fit_int(B, capacity, heads)) return ASR_ERR_UNSUPPORTED;
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

// The append + self step, with or without a beam reorder (idx != nullptr:
// kv is the source cache, cache_w the destination, lens the source lengths).
static int self_append_step(const float* q, int64_t q_stride, const float* k_new,
                            const float* v_new, int64_t kv_stride, const uint16_t* src,
                            uint16_t* cache, int64_t seq_stride, const int32_t* idx,
                            const int32_t* lens, int32_t* lens_out, int B, int heads,
                            int head_dim, int capacity, float scale, float* out, void* ws,
                            size_t ws_bytes, int32_t* dev_err, cudaStream_t stream) {
  if (B < 0 || B > ASR_MAX_BATCH || heads < 1 || capacity < 1) return ASR_ERR_INVALID_ARG;
  if ((head_dim != 64 && head_dim != 128) || heads > ASR_MAX_KV_HEADS) return ASR_ERR_UNSUPPORTED;
  if (B == 0) return ASR_OK;
  if (!q || !k_new || !v_new || !src || !cache || !lens || !out) return ASR_ERR_INVALID_ARG;
  const int64_t row = 2LL * heads * head_dim;
  if (q_stride < (int64_t)heads * head_dim || kv_stride < (int64_t)heads * head_dim ||
      seq_stride < (int64_t)capacity * row)
    return ASR_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(src) ||
      !aligned16(cache) || !aligned16(out) || q_stride % 4 != 0 || kv_stride % 4 != 0 ||
      seq_stride % 8 != 0)
    return ASR_ERR_MISALIGNED;
  if (!rows_fit_int(B, capacity, heads)) return ASR_ERR_UNSUPPORTED;
  if (idx) {
    // the destination rows must not overlap the source rows, and lens_out
    // neither the lengths nor the indices (other CTAs still read them)
    const uintptr_t bytes = ((uintptr_t)(B - 1) * (uintptr_t)seq_stride +
                             (uintptr_t)capacity * (uintptr_t)row) * 2;
    const uintptr_t s0 = (uintptr_t)src, d0 = (uintptr_t)cache;
    if (s0 < d0 + bytes && d0 < s0 + bytes) return ASR_ERR_ALIAS;
    const uintptr_t ib = (uintptr_t)B * 4, o0 = (uintptr_t)lens_out;
    const uintptr_t l0 = (uintptr_t)lens, x0 = (uintptr_t)idx;
    if ((o0 < l0 + ib && l0 < o0 + ib) || (o0 < x0 + ib && x0 < o0 + ib)) return ASR_ERR_ALIAS;
  }
  DecodeArgs a = {};
  a.q = q;
  a.q_stride = q_stride;
  a.kv = src;
  a.cache_w = cache;
  a.src_stride = seq_stride;
  a.row_elems = (int)row;
  a.n_src = B;
  a.B = B;
  a.lens = lens;
  a.idx = idx;
  a.lens_out = lens_out;
  a.capacity = capacity;
  a.Hq = heads;
  a.Hkv = heads;
  a.rep = 1;
  a.max_members = 1;
  a.qscale = scale * kLog2e;
  a.out = out;
  a.dev_err = dev_err;
  a.mode = kModeSelf;
  a.append = 1;
  a.kv_stride = kv_stride;
  a.k_new = k_new;
  a.v_new = v_new;
  return launch_decode(a, head_dim, 1, ws, ws_bytes, stream);
}

extern "C" int asr_self_attn_append_step(const float* q, int64_t q_stride, const float* k_new,
                                         const float* v_new, int64_t kv_stride, uint16_t* cache,
                                         int64_t seq_stride, const int32_t* lens, int B, int heads,
                                         int head_dim, int capacity, float scale, float* out,
                                         void* ws, size_t ws_bytes, int32_t* dev_err,
                                         asr_stream_t stream) {
  return self_append_step(q, q_stride, k_new, v_new, kv_stride, cache, cache, seq_stride, nullptr,
                          lens, nullptr, B, heads, head_dim, capacity, scale, out, ws, ws_bytes,
                          dev_err, (cudaStream_t)stream);
}

extern "C" int asr_self_attn_reorder_append_step(
    const float* q, int64_t q_stride, const float* k_new, const float* v_new, int64_t kv_stride,
    const uint16_t* cache_src, uint16_t* cache_dst, int64_t seq_stride, const int32_t* idx,
    const int32_t* lens_src, int32_t* lens_dst, int B, int heads, int head_dim, int capacity,
    float scale, float* out, void* ws, size_t ws_bytes, int32_t* dev_err, asr_stream_t stream) {
  if (B > 0 && (!idx || !lens_dst)) return ASR_ERR_INVALID_ARG;
  return self_append_step(q, q_stride, k_new, v_new, kv_stride, cache_src, cache_dst, seq_stride,
                          idx, lens_src, lens_dst, B, heads, head_dim, capacity, scale, out, ws,
                          ws_bytes, dev_err, (cudaStream_t)stream);
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
  if (!rows_fit_int(G, frames, heads)) return ASR_ERR_UNSUPPORTED;
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

extern "C" int asr_gqa_step(const float* q, int64_t q_stride, const float* k_new,
                            const float* v_new, int64_t kv_stride, const float* q_norm_w,
                            const float* k_norm_w, float eps, float rope_base,
                            const int32_t* n_past, uint16_t* cache,
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
  if (seq_stride < (int64_t)capacity * row || q_stride < (int64_t)q_heads * head_dim ||
      kv_stride < (int64_t)kv_heads * head_dim)
    return ASR_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(q_norm_w) ||
      !aligned16(k_norm_w) || !aligned16(cache) || !aligned16(out) || seq_stride % 8 != 0 ||
      q_stride % 4 != 0 || kv_stride % 4 != 0)
    return ASR_ERR_MISALIGNED;
  if (!rows_fit_int(B, capacity, kv_heads)) return ASR_ERR_UNSUPPORTED;
  DecodeArgs a = {};
  a.q = q;
  a.q_stride = q_stride;
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
  a.append = 1;
  a.kv_stride = kv_stride;
  a.k_new = k_new;
  a.v_new = v_new;
  a.wq = q_norm_w;
  a.wk = k_norm_w;
  a.eps = eps;
  for (int i = 0; i < head_dim / 2; ++i) {
    // theta_i / (2 pi) as a float pair hi + lo
    const double t = pow((double)rope_base, -2.0 * i / head_dim) / (2.0 * 3.14159265358979323846);
    const float hi = (float)t;
    a.rope_turns[2 * i] = hi;
    a.rope_turns[2 * i + 1] = (float)(t - (double)hi);
  }
  return launch_decode(a, head_dim, a.rep, ws, ws_bytes, (cudaStream_t)stream);
}
