// decode_attn.cuh -- shared definitions of the split-K decode-attention kernel
// (kernel in decode_attn.cu, workspace sizing in abi.cu).
#pragma once

#include <cuda.h>
#include <stddef.h>
#include <stdint.h>

namespace asrkv {

enum DecodeMode { kModeSelf = 0, kModeCross = 1, kModeGqa = 2 };

// Most persistent CTAs per SM any decode launch uses; bounds the number of
// partial results a workspace must hold.
constexpr int kMaxCtasPerSm = 4;

// Rows per box of the large tensor-map copy of a head group's row chunks.
constexpr int kBoxRows = 8;

struct DecodeArgs {
  // tensor maps of the K/V rows, used when a work unit is a group of KV heads
  // narrower than the row (HS > 1): dims {HD, Hkv, 2 (K, V), rows, sources},
  // boxes {HD, hs, 2, kBoxRows or 1, 1}
  CUtensorMap tmap_rows;
  CUtensorMap tmap_row;
  // queries: fp32, sequence b at q + b*q_stride, head h at h*HD
  const float* q;
  int64_t q_stride;
  // keys/values: f16 rows (K of all KV heads, then V), source g at kv + g*src_stride
  const uint16_t* kv;
  int64_t src_stride;
  int row_elems;
  int n_src;  // sources: sequences (self, GQA) or groups (cross)
  int B;      // query sequences
  const int32_t* lens;   // self: keys per sequence; GQA: n_past per sequence
  const int32_t* group;  // cross: source of each sequence (non-decreasing)
  int fixed_len;         // cross: frames per source
  int capacity;          // self / GQA: rows per sequence cache
  int Hq, Hkv, rep;      // rep = Hq / Hkv
  int max_members;       // cross: max sequences per group; else 1
  float qscale;          // scale * log2(e): scores are kept in the log2 domain
  float* out;            // fp32 [B][Hq*HD]
  // work units: source g is split into HS groups of hs = Hkv / HS KV heads;
  // unit u = g * HS + hg streams the hs heads' K and V chunks of g's rows
  int HS, hs;
  int chunk_elems;  // f16 elements of one row chunk in shared memory (2 * hs * HD)
  int n_units;      // n_src * HS
  // workspace
  int* counters;   // [n_units], zero between calls
  float* part_ml;  // [(P + n_units) * max_members * hs * rep][2]  (max, sum) per partial
  float* part_o;   // [(P + n_units) * max_members * hs * rep][HD] unnormalised output
  int32_t* dev_err;
  // tiling
  int R;            // row slots (groups of the same head working on different rows)
  int MS;           // query splits: groups of one head and row slot, each on NQ of its queries
  int tile_rows;    // rows per pipeline stage (R * rows per slot)
  int min_share;    // fewest rows one CTA takes (bounds the partials per unit)
  int seg_rows;     // virtual rows charged per unit on the flattened key axis
  int stages;       // pipeline depth
  int stage_elems;  // f16 elements per stage buffer (128-byte multiple)
  int mode;         // DecodeMode
  int pf_bytes;     // K/V bytes of its share a CTA asks L2 to prefetch before the grid dependency wait
  uint64_t wait_ns; // bound of every mbarrier wait (ns of %globaltimer)
  int stall;        // test support: the producer issues no copies, so every wait runs out
  int early;        // the caller promised the lengths and history are ready (asr_set_history_ready)
  // new-token append (GQA step, fused self step): the call writes row p and
  // folds that key in; p = n_past (GQA) or lens - 1 (self)
  int append;
  int64_t kv_stride;  // floats between sequences of k_new / v_new
  const float* k_new;
  const float* v_new;
  // self step with a beam reorder (take along the batch axis, fused): source
  // g streams the history rows of sequence idx[g] of kv and stores them to
  // sequence g of cache_w (same strides) as they pass through shared memory;
  // lens holds the source lengths and lens_out[g] = lens[idx[g]] (0 when
  // sequence g is skipped).  idx == nullptr: no reorder.
  const int32_t* idx;
  int32_t* lens_out;
  // GQA only
  const float* wq;
  const float* wk;
  float eps;
  uint16_t* cache_w;  // the cache, writable (row p is appended)
  float rope_turns[128];  // theta_i / (2 pi) as float pairs (hi, lo), theta_i = rope_base^(-2i/HD), i < HD/2
};

// Shared-memory layout of one CTA (bytes from the dynamic smem base).
//   bars: full/empty mbarriers of the stage ring; ctl: control words; off,
//     mstart: the consumers' source offsets and first sequences; poff, psrc:
//     the producer's offsets and the cache sequence each source reads (beam
//     reorder); slen: the length entry of each source (self,
//     GQA); rope, wts: GQA tables; merge: the row slots' states (R entries
//     of Hv x NQ); stage: the K/V ring.
struct DecodeSmem {
  int bars, ctl, off, mstart, poff, psrc, slen, rope, wts, merge, stage, total;
};

__host__ __device__ inline int dsm_align(int x, int a) { return (x + a - 1) / a * a; }

// Hv: virtual heads of a unit (query splits x KV heads of the group).
__host__ __device__ inline DecodeSmem decode_smem_layout(int stages, int n_src, int R, int Hv,
                                                         int NQ, int HD, int stage_elems) {
  DecodeSmem s;
  s.bars = 0;
  s.ctl = dsm_align(s.bars + 2 * stages * 8, 16);
  s.off = dsm_align(s.ctl + 16 * 4, 16);
  s.mstart = dsm_align(s.off + (n_src + 1) * 4, 16);
  s.poff = dsm_align(s.mstart + (n_src + 1) * 4, 16);
  s.psrc = dsm_align(s.poff + (n_src + 1) * 4, 16);
  s.slen = dsm_align(s.psrc + (n_src + 1) * 4, 16);
  s.rope = dsm_align(s.slen + (n_src + 1) * 4, 16);
  s.wts = dsm_align(s.rope + (HD > 64 ? HD : 64) * 4, 16);
  s.merge = dsm_align(s.wts + 2 * HD * 4, 16);
  s.stage = dsm_align(s.merge + R * Hv * NQ * (HD + 4) * 4, 128);
  s.total = s.stage + stages * stage_elems * 2;
  return s;
}

// Workspace bytes of a decode call with n_src sources and Hq query heads on a
// device with `sms` SMs (any head split: a unit of hs KV heads keeps only
// its own query heads' partials).
size_t decode_ws_bytes(int n_src, int max_members, int Hq, int HD, int sms);

// Bytes at the start of that workspace that hold the per-unit counters (zero
// between calls).
size_t decode_counter_bytes(int n_src, int Hq);

}  // namespace asrkv
