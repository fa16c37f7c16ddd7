/*
 * asrkv.h -- C ABI of libasrkv.so: GB300 (sm_103a) kernels for the per-token
 * decoder step of encoder-decoder speech recognisers (Whisper-style MHA and a
 * Qwen3-ASR-style GQA decoder) over f16 K/V caches.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All data pointers are DEVICE pointers owned by the caller.  The library
 *    keeps no pointer after a call returns and allocates no device memory.
 *  - f16 data are IEEE binary16 bit patterns passed as uint16_t*.
 *  - A cache ROW holds 2*Hkv*hd f16: the K vectors of KV heads 0..Hkv-1, then
 *    the V vectors of KV heads 0..Hkv-1; head h sits at offset h*hd inside its
 *    half ("wavo 0.1.0, src/whisper/decoder.rs", doc of `Buffers`: a cache row
 *    is K then V of all heads, as f16).  Rows of one sequence are contiguous.
 *  - Query head h reads KV head h / (Hq/Hkv) (contiguous GQA groups).
 *  - Every call is asynchronous on `stream` (NULL = the legacy default
 *    stream), never synchronises, and returns an asr_status.  All argument
 *    checks happen on the host before anything is enqueued; a call that
 *    returns an error has enqueued nothing.
 *  - Data errors found on the device (a length or index out of range) never
 *    trap: the affected sequence is skipped (its output row is set to 0 where
 *    the call has one) and an ASR_DEVERR_* bit is OR-ed into *dev_err when
 *    dev_err is not NULL.  The caller zeroes *dev_err and reads it back.
 *  - Per-step scalars (lengths, positions, slots, indices) live in device
 *    arrays, so a whole decode step can be captured once in a CUDA graph and
 *    replayed; the graph's shape depends only on capacities ("transcribe.cpp,
 *    src/arch/qwen3_asr/decoder.h", comment of build_step_graph: a static step
 *    graph reused across steps).
 *  - Attention scores are scale * (q . k) in fp32, softmax in fp32, output
 *    fp32.  The caller passes `scale`; the pages use (D/H)^-0.5 = hd^-0.5
 *    ("Nest whisper-tiny, src/lib.linnet", Attention.attend: rsqrt(D/Heads)).
 *
 * Workspace: the attention entry points split long key ranges over many CTAs
 * and merge the pieces (flash-decoding with a log-sum-exp combine).  They
 * need a caller-provided workspace of at least asr_workspace_size(...) bytes,
 * 256-byte aligned, ZERO-FILLED before its first use (cudaMemsetAsync).  Each
 * call leaves the workspace's counters at zero again, so one zeroing at
 * allocation time is enough; a workspace must not be shared by calls that can
 * run concurrently (different streams without ordering).
 */
#ifndef ASRKV_H
#define ASRKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* asr_stream_t;

/* Return codes. */
enum asr_status {
  ASR_OK = 0,
  ASR_ERR_INVALID_ARG = 1, /* NULL pointer, size out of range, stride too small */
  ASR_ERR_UNSUPPORTED = 2, /* head_dim not 64/128, Hq % Hkv != 0, too many heads/beams/sequences */
  ASR_ERR_MISALIGNED = 3,  /* a pointer or stride is not 16-byte aligned */
  ASR_ERR_ALIAS = 4,       /* rearrange source and destination overlap */
  ASR_ERR_WORKSPACE = 5,   /* workspace NULL, too small or not 256-byte aligned */
  ASR_ERR_CUDA = 6,        /* a CUDA runtime call or launch failed */
  ASR_ERR_SCRATCH_LIMIT = 7, /* the problem needs more scratch than the library's fixed array */
};

/* Bits OR-ed into *dev_err by the kernels. */
#define ASR_DEVERR_LEN 0x1     /* a length / position / slot outside its range */
#define ASR_DEVERR_INDEX 0x2   /* a beam index or group id outside its range, or groups not sorted */
#define ASR_DEVERR_BEAMS 0x4   /* a group has more sequences than max_beams */
#define ASR_DEVERR_TIMEOUT 0x8 /* a bounded wait inside a kernel gave up (never expected) */

/* Operation ids for asr_workspace_size. */
enum asr_op {
  ASR_OP_SELF_ATTN = 1,
  ASR_OP_CROSS_ATTN = 2,
  ASR_OP_GQA_STEP = 3,
  ASR_OP_PREFILL_ATTN = 4,
  ASR_OP_MHA_PREFILL = 5,
  ASR_OP_ENCODER_ATTN = 6,
};

/* Epilogues of asr_linear. */
enum asr_linear_mode {
  ASR_LINEAR_STORE = 0,    /* y = v            (wavo's Epilogue::Bias) */
  ASR_LINEAR_RESIDUAL = 1, /* y = y + v        (Epilogue::Residual(1.0)) */
  ASR_LINEAR_GELU = 2,     /* y = v * Phi(v)   (Epilogue::Gelu, the erf form) */
};

/* Pre-norms of asr_linear. */
enum asr_norm {
  ASR_NORM_NONE = 0,
  ASR_NORM_LAYER = 1, /* LayerNorm: (x - mean) / sqrt(var + eps) * w + b */
  ASR_NORM_RMS = 2,   /* RMSNorm:   x / sqrt(mean(x^2) + eps) * w */
};

/* Input activations of asr_linear. */
enum asr_act {
  ASR_ACT_NONE = 0,
  ASR_ACT_SWIGLU = 1, /* a_k = silu(x_k) * x_{K+k}: rows hold [gate | up], 2K values */
};

/* Limits checked on the host. */
#define ASR_MAX_BATCH 2048 /* sequences (and groups) per call */
#define ASR_MAX_BEAMS 8    /* sequences sharing one cross source; also max Hq/Hkv */
#define ASR_MAX_KV_HEADS 64

/* a1 -- K/V append.
 * Defines: "wavo 0.1.0, src/whisper/decoder.rs", Decoder::record_step (k and v
 * of the new token packed as f16 into cache row `pos`); "Nest whisper-tiny,
 * src/lib.linnet", DecoderLayer.step (write_at(self_k/self_v, ..., pos)).
 *   cache[b*seq_stride + slot[b]*row + i] = f16_rne(k[b*src_row_stride + i])      i < Hkv*hd
 *   cache[b*seq_stride + slot[b]*row + Hkv*hd + i] = f16_rne(v[b*src_row_stride + i])
 * with row = 2*kv_heads*head_dim; f16_rne is IEEE round to nearest even with
 * overflow to infinity.  k, v: fp32 [B][src_row_stride] (e.g. the k and v
 * parts of a [q|k|v] projection row, src_row_stride = 3*d); slot: int32 [B],
 * device.  A slot outside [0, capacity) skips that sequence (ASR_DEVERR_LEN).
 * Alignment: k, v, cache 16-byte aligned; src_row_stride % 4 == 0;
 * seq_stride % 8 == 0 and >= capacity*row.  head_dim % 8 == 0. */
int asr_kv_append(const float* k, const float* v, int64_t src_row_stride, uint16_t* cache,
                  int64_t seq_stride, const int32_t* slot, int B, int kv_heads, int head_dim,
                  int capacity, int32_t* dev_err, asr_stream_t stream);

/* a2 (+ a4) -- causal self-attention of one new token per sequence.
 * Defines: "wavo 0.1.0, src/whisper/decoder.rs", Decoder::record_step
 * (attend(q, own, pos+1)); "Nest whisper-tiny, src/lib.linnet",
 * DecoderLayer.step (mask: slots <= pos); "mlx-bun whisper.ts", #attention
 * (additive causal mask, precise softmax).
 *   For sequence b and head h, with L = lens[b] keys (the new token's own key,
 *   appended before this call, is row L-1):
 *   z_j = scale * q_bh . K_bj,h  (j < L);  out_bh = sum_j softmax(z)_j V_bj,h
 * q: fp32 [B][q_stride] (head h at h*head_dim); cache: f16 [B][seq_stride]
 * rows as above with Hkv = heads; lens: int32 [B], device, each in
 * [1, capacity] (else the row of out is zeroed, ASR_DEVERR_LEN); out: fp32
 * [B][heads*head_dim], contiguous.  head_dim in {64, 128}; heads <= 64;
 * B <= ASR_MAX_BATCH.  q_stride % 4 == 0; seq_stride % 8 == 0.
 * ws: workspace of asr_workspace_size(ASR_OP_SELF_ATTN, B, B, 1, heads, head_dim, 0) bytes. */
int asr_self_attn_step(const float* q, int64_t q_stride, const uint16_t* cache,
                       int64_t seq_stride, const int32_t* lens, int B, int heads, int head_dim,
                       int capacity, float scale, float* out, void* ws, size_t ws_bytes,
                       int32_t* dev_err, asr_stream_t stream);

/* a1 + a2 (+ a4) fused -- append the new token's K/V and attend, in one launch.
 * Same definitions as asr_kv_append followed by asr_self_attn_step: row
 * lens[b]-1 of sequence b becomes f16_rne(k_new_b) || f16_rne(v_new_b) and the
 * token attends rows [0, lens[b]) ("wavo 0.1.0, src/whisper/decoder.rs",
 * Decoder::record_step: pack k,v into row pos, then attend over pos+1 rows).
 * The cache bytes written are identical to those of asr_kv_append; the key
 * of the new row is taken from the rounded k_new rather than re-read.
 * k_new, v_new: fp32 [B][kv_stride] (the k and v parts of [q|k|v] rows:
 * kv_stride = 3*d, v_new = k_new + d); kv_stride % 4 == 0.  Other arguments
 * and errors as asr_self_attn_step (lens outside [1, capacity]: output
 * zeroed, nothing written).  ws: the ASR_OP_SELF_ATTN size. */
int asr_self_attn_append_step(const float* q, int64_t q_stride, const float* k_new,
                              const float* v_new, int64_t kv_stride, uint16_t* cache,
                              int64_t seq_stride, const int32_t* lens, int B, int heads,
                              int head_dim, int capacity, float scale, float* out, void* ws,
                              size_t ws_bytes, int32_t* dev_err, asr_stream_t stream);

/* a6 + a1 + a2 fused -- beam reorder of one layer's self cache, append of the
 * new token and self-attention, in one launch.
 * Defines: "mlx-bun whisper.ts", WhisperKvCache.rearrange (take along the batch
 * axis of the self k/v before the step) followed by the append + self step
 * above.  Equal, byte for byte in cache_dst and lens_dst and in out, to
 * asr_kv_rearrange over this one layer (n_layers = 1) followed by
 * asr_self_attn_append_step on cache_dst with lens = lens_dst:
 *   for beam b with s = idx[b] and L = lens_src[s]:
 *   rows [0, L-1) of cache_dst[b] = rows [0, L-1) of cache_src[s] (bitwise);
 *   row L-1 of cache_dst[b] = f16_rne(k_new_b) || f16_rne(v_new_b);
 *   out_b = self-attention of q_b over rows [0, L) of cache_dst[b];
 *   lens_dst[b] = L.
 * The history rows are read once: each tile is attended from shared memory
 * and stored to cache_dst from there.  idx, lens_src, lens_dst: int32 [B],
 * device.  idx[b] outside [0, B) (ASR_DEVERR_INDEX) or L outside
 * [1, capacity] (ASR_DEVERR_LEN) skips beam b: its output row is zeroed,
 * lens_dst[b] = 0 and cache_dst[b] is left untouched.  cache_src and
 * cache_dst share seq_stride and must not overlap (ASR_ERR_ALIAS), nor may
 * lens_dst overlap lens_src or idx.  Rows of cache_dst past L are left
 * untouched.  Other arguments, alignment and errors as
 * asr_self_attn_append_step; ws: the ASR_OP_SELF_ATTN size. */
int asr_self_attn_reorder_append_step(const float* q, int64_t q_stride, const float* k_new,
                                      const float* v_new, int64_t kv_stride,
                                      const uint16_t* cache_src, uint16_t* cache_dst,
                                      int64_t seq_stride, const int32_t* idx,
                                      const int32_t* lens_src, int32_t* lens_dst, int B,
                                      int heads, int head_dim, int capacity, float scale,
                                      float* out, void* ws, size_t ws_bytes, int32_t* dev_err,
                                      asr_stream_t stream);

/* a3 (+ a4) -- cross-attention of one token per sequence over the encoder's
 * cached K/V, shared by the beams of one audio.
 * Defines: "wavo 0.1.0, src/whisper/decoder.rs", Decoder::record_step
 * (attend(q, cross, frames)); "Nest whisper-tiny, src/lib.linnet",
 * DecoderLayer.cross (no mask); "mlx-bun whisper.ts", #attention (k/v keep
 * their own batch: beams attend one broadcast encoder output).
 *   Sequence b attends all `frames` rows of source group[b]:
 *   out_bh = sum_j softmax_j(scale * q_bh . K_{group[b]} j,h) V_{group[b]} j,h
 * cross: f16 [G][group_stride] rows with Hkv = heads; group: int32 [B],
 * device, NON-DECREASING (the beams of one audio are consecutive), each in
 * [0, G) (else the output row is zeroed, ASR_DEVERR_INDEX); at most
 * max_beams (<= ASR_MAX_BEAMS) sequences per group (extra ones are zeroed,
 * ASR_DEVERR_BEAMS).  Each group's K/V is read once for all its beams.
 * ws: asr_workspace_size(ASR_OP_CROSS_ATTN, B, G, max_beams, heads, head_dim, 0) bytes. */
int asr_cross_attn_step(const float* q, int64_t q_stride, const uint16_t* cross,
                        int64_t group_stride, const int32_t* group, int B, int G, int max_beams,
                        int heads, int head_dim, int frames, float scale, float* out, void* ws,
                        size_t ws_bytes, int32_t* dev_err, asr_stream_t stream);

/* a5 -- Qwen3-ASR-style GQA decode step, fused: per-head Q/K RMSNorm, NeoX
 * RoPE, K/V append and grouped-query attention.
 * Defines: "transcribe.cpp, src/arch/qwen3_asr/decoder.h", header comment
 * (RMSNorm weight*rsqrt(mean(x^2)+eps)*x; per-head Q/K RMSNorm over head_dim
 * after projection and before RoPE; NeoX rotate_half RoPE at freq_base 1e6;
 * GQA 16 Q / 8 KV heads of 128) and StepBuildBatched (position = n_past, K/V
 * written at row n_past, positions > n_past masked).
 *   For sequence b at p = n_past[b]:
 *   k^_h = RoPE_p(RMSNorm(k_new_bh) * k_norm_w);  q^_h = RoPE_p(RMSNorm(q_bh) * q_norm_w)
 *   cache row p = f16(k^) || f16(v_new_b)                    (written by this call)
 *   out_bh = attention of q^_h over rows [0, p] of KV head h / (Hq/Hkv)
 *   RoPE_p turns the pair (i, i + hd/2) by p * rope_base^(-2i/hd).
 * q: fp32 [B][q_stride] (q_heads*hd used); k_new, v_new: fp32 [B][kv_stride]
 * (kv_heads*hd used; one stride for both; strides % 4 == 0); q_norm_w,
 * k_norm_w: fp32 [hd] (shared by all heads); n_past: int32 [B], device, in
 * [0, capacity) (else output zeroed, cache untouched, ASR_DEVERR_LEN);
 * out: fp32 [B][q_heads*hd].  head_dim in {64, 128}; q_heads % kv_heads == 0;
 * q_heads/kv_heads <= ASR_MAX_BEAMS.
 * ws: asr_workspace_size(ASR_OP_GQA_STEP, B, B, 1, q_heads, head_dim, 0) bytes. */
int asr_gqa_step(const float* q, int64_t q_stride, const float* k_new, const float* v_new,
                 int64_t kv_stride, const float* q_norm_w, const float* k_norm_w, float eps,
                 float rope_base, const int32_t* n_past,
                 uint16_t* cache, int64_t seq_stride, int capacity, int B, int q_heads,
                 int kv_heads, int head_dim, float scale, float* out, void* ws, size_t ws_bytes,
                 int32_t* dev_err, asr_stream_t stream);

/* a6 -- beam reorder of the self caches of n_layers layers.
 * Defines: "mlx-bun whisper.ts", WhisperKvCache.rearrange (take along the batch
 * axis of every layer's self k/v; cross k/v broadcast from one audio are left
 * alone).
 *   For each beam b with s = idx[b]: the n = lens_src[s] - 1 history rows
 *   (the rows written before the coming step's token) of every layer l are
 *   copied, dst[b*seq_stride + l*layer_stride + 0 .. n*row_elems) =
 *              src[s*seq_stride + l*layer_stride + 0 .. n*row_elems),
 *   and lens_dst[b] = lens_src[s].  Rows past n are left untouched.
 * idx, lens_src, lens_dst: int32 [B], device.  idx outside [0, B) or
 * lens_src[s] outside [1, capacity] skips the beam with lens_dst[b] = 0
 * (ASR_DEVERR_INDEX / ASR_DEVERR_LEN).  src and dst must not overlap
 * (ASR_ERR_ALIAS).  row_elems % 8 == 0; strides % 8 == 0; pointers 16-byte
 * aligned; B * n_layers <= 65535.  Copies are bitwise. */
int asr_kv_rearrange(const uint16_t* src, uint16_t* dst, int64_t seq_stride, int64_t layer_stride,
                     int n_layers, int row_elems, int capacity, const int32_t* idx,
                     const int32_t* lens_src, int32_t* lens_dst, int B, int32_t* dev_err,
                     asr_stream_t stream);

/* a7 + a8 -- batched causal prefill of a Qwen3-ASR-style decoder.
 * Defines: "transcribe.cpp, src/arch/qwen3_asr/decoder.h", header comment
 * (per-head Q/K RMSNorm after projection and before RoPE; NeoX RoPE at
 * freq_base 1e6; GQA) and PrefillBuildBatched (positions shared 0..T-1, K/V
 * written to cache rows [0, T), shared causal mask); "Nest whisper-tiny,
 * src/lib.linnet", DecoderLayer.prefill (write_span at 0, causal mask).
 *   For every sequence b and position t < T:
 *   q^_t,h = f16(RoPE_t(RMSNorm(q_t,h) * q_norm_w)), k^_t,h likewise with k_norm_w;
 *   cache row t = k^_t || v_t  (v copied bitwise);
 *   out_t,h = sum_{j<=t} softmax_j(scale * q^_t,h . k^_j,kvh(h)) v_j,kvh(h)
 * The f16 rounding of q^ and k^ is part of the operation (they are the
 * tensor-core operands); the softmax weights enter the P.V product as f16.
 * q: f16 [B][T][q_heads*128]; k, v: f16 [B][T][kv_heads*128]; q_norm_w,
 * k_norm_w: fp32 [128]; cache: f16 [B][seq_stride] (rows of 2*kv_heads*128);
 * out: fp32 [B][T][q_heads*128].  head_dim must be 128; kv_heads <= 16;
 * q_heads % kv_heads == 0; T <= capacity.  Runs on the tensor cores
 * (tcgen05); needs an sm_100-family GPU.
 * ws: asr_workspace_size(ASR_OP_PREFILL_ATTN, B, kv_heads, 1, q_heads, 128, T)
 * bytes (n_sources = kv_heads for this op); need not be zeroed. */
int asr_prefill_attn(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                     const float* q_norm_w, const float* k_norm_w, float eps, float rope_base,
                     int B, int T, int q_heads, int kv_heads, int head_dim, float scale,
                     uint16_t* cache, int64_t seq_stride, int capacity, float* out, void* ws,
                     size_t ws_bytes, int32_t* dev_err, asr_stream_t stream);

/* a7 alone -- the prefill preparation of asr_prefill_attn: cache rows [0, T)
 * (roped K, V) and, in the workspace, q^ for the tensor cores.  Same
 * arguments and definitions as asr_prefill_attn. */
int asr_prefill_prep(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                     const float* q_norm_w, const float* k_norm_w, float eps, float rope_base,
                     int B, int T, int q_heads, int kv_heads, int head_dim, uint16_t* cache,
                     int64_t seq_stride, int capacity, void* ws, size_t ws_bytes,
                     asr_stream_t stream);

/* a8 alone -- the causal attention of asr_prefill_attn, reading what
 * asr_prefill_prep left in the cache and the workspace (same workspace,
 * unchanged in between). */
int asr_prefill_attention(int B, int T, int q_heads, int kv_heads, int head_dim, float scale,
                          const uint16_t* cache, int64_t seq_stride, int capacity, float* out,
                          void* ws, size_t ws_bytes, int32_t* dev_err, asr_stream_t stream);

/* Next row -- batched multi-head prompt prefill with per-sequence lengths.
 * Defines: "Nest whisper-tiny, src/lib.linnet", DecoderLayer.prefill (the S
 * prompt tokens' keys and values go to the self cache at rows [0, S); they
 * attend causally among themselves); "transcribe.cpp, src/arch/qwen3_asr/
 * decoder.h", PrefillBuildBatched (prompts of up to T_prompt_max tokens,
 * each with its own last real position).
 *   For each sequence b with L = lens[b] (lens NULL: L = T) and t < L:
 *   cache row t = k_t || v_t (bitwise, all heads);
 *   out_t,h = sum_{j<=t} softmax_j(scale * q_t,h . k_j,h) v_j,h
 *   Rows t >= L of out and of the cache are not written.
 * q, k, v: f16 [B][T][heads*head_dim] (heads = KV heads: multi-head); lens:
 * int32 [B] device or NULL; a length outside [0, T] skips the sequence
 * (ASR_DEVERR_LEN).  cache: f16 [B][seq_stride], rows of 2*heads*head_dim;
 * T <= capacity.  out: fp32 [B][T][heads*head_dim].  head_dim 64 or 128;
 * heads <= ASR_MAX_KV_HEADS.  The softmax weights enter the P.V product as
 * f16 (tensor cores, tcgen05).
 * ws: asr_workspace_size(ASR_OP_MHA_PREFILL, B, heads, 1, heads, head_dim, T)
 * bytes (V transposed, used when lens is given); need not be zeroed. */
int asr_mha_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v, const int32_t* lens,
                    int B, int T, int heads, int head_dim, float scale, uint16_t* cache,
                    int64_t seq_stride, int capacity, float* out, void* ws, size_t ws_bytes,
                    int32_t* dev_err, asr_stream_t stream);

/* Next row -- the encoder's self-attention over its frames, unmasked.
 * Defines: "Nest whisper-tiny, src/lib.linnet", EncoderLayer.forward (every
 * audio position attends to every other, the padding of the fixed 30 s
 * included; no mask); "mlx-bun whisper.ts", the encoder blocks' #attention
 * (no mask).
 *   For each sequence b with L = lens[b] (lens NULL: L = T) and t < L:
 *   out_t,h = sum_{j<L} softmax_j(scale * q_t,h . k_j,h) v_j,h
 *   Rows t >= L of out are not written.
 * Same arrays, limits and errors as asr_mha_prefill, without the cache.
 * ws: asr_workspace_size(ASR_OP_ENCODER_ATTN, B, heads, 1, heads, head_dim, T)
 * bytes; need not be zeroed. */
int asr_encoder_attn(const uint16_t* q, const uint16_t* k, const uint16_t* v, const int32_t* lens,
                     int B, int T, int heads, int head_dim, float scale, float* out, void* ws,
                     size_t ws_bytes, int32_t* dev_err, asr_stream_t stream);

/* Next row -- the cross-attention K/V of one decoder layer from the encoder
 * output.  Defines: "wavo 0.1.0, src/whisper/decoder.rs",
 * Decoder::record_cross (a GEMM of the encoder rows with the layer's [k | v]
 * weight and a bias epilogue, then a pack to f16 cache rows) and
 * Decoder::load (k has no bias; v has its own); "Nest whisper-tiny,
 * src/lib.linnet", DecoderLayer.listen.
 *   For each group g and frame t < frames, cross row t of group g:
 *   element n = f16( sum_k enc[g][t][k] * w[n][k] + (n >= d ? bias_v[n-d] : 0) )
 *   i.e. K of all heads in elements [0, d), V in [d, 2d) -- the row the
 *   cross-attention step reads.  Rows at and past `frames` are not written.
 * enc: f16 [G][frames][d]; w: f16 [2d][d] (row n produces element n); bias_v:
 * fp32 [d]; cross: f16 [G][group_stride], group_stride >= frames * 2d.
 * d % 128 == 0 (Whisper: 384, 512, 768, 1024, 1280).  The products run on
 * the tensor cores (tcgen05, f16 operands, fp32 accumulation); the bias is
 * added in fp32 and the result rounded to nearest even.  No workspace. */
int asr_cross_kv_fill(const uint16_t* enc, const uint16_t* w, const float* bias_v, int G,
                      int frames, int d, uint16_t* cross, int64_t group_stride, int32_t* dev_err,
                      asr_stream_t stream);

/* Next row -- one dense step of a decoder layer around the attention.
 * Defines: "wavo 0.1.0, src/whisper/decoder.rs", Decoder::record_step
 * (layer_norm of x, then gemv with the layer's qkv / self_out / cross_q /
 * cross_out / fc1 / fc2 weight and the epilogue Bias, Residual(1.0) or
 * Gelu); "Nest whisper-tiny, src/lib.linnet", LayerNorm (torch.nn.LayerNorm,
 * eps 1e-5) and Mlp (fc2(gelu_erf(fc1(x)))); "transcribe.cpp,
 * src/arch/qwen3_asr/decoder.h", header comment (pre-norm RMSNorm
 * weight * rsqrt(mean(x^2) + eps) * x; SwiGLU MLP down(silu(gate(x)) * up(x))).
 *   a_m  = x_m                                  norm ASR_NORM_NONE
 *        = (x_m - mean_m) / sqrt(var_m + eps) * norm_w + norm_b   ASR_NORM_LAYER
 *          (mean and biased variance over the K values of row m)
 *        = x_m / sqrt(mean_k x_mk^2 + eps) * norm_w                ASR_NORM_RMS
 *   with act ASR_ACT_SWIGLU (no norm): a_mk = silu(x_mk) * x_m,K+k, silu(v) =
 *   v / (1 + e^-v): the row holds the gate half then the up half.
 *   v_mn = sum_k a_mk * w[n][k] + bias[n]                     (bias NULL: 0)
 *   y_mn = v_mn (ASR_LINEAR_STORE) | y_mn + v_mn (ASR_LINEAR_RESIDUAL)
 *        | v_mn * Phi(v_mn) = v/2 (1 + erf(v/sqrt 2)) (ASR_LINEAR_GELU)
 * x: fp32 [M][x_stride] (the first K values used, 2K with SwiGLU; 16-byte
 * aligned, x_stride % 4 == 0); norm_w, norm_b: fp32 [K] (16-byte aligned;
 * norm_b only for LayerNorm); w: f16 [N][K] (row n makes output n: torch's
 * Linear layout; 16-byte aligned); bias: fp32 [N] or NULL; y: fp32
 * [M][y_stride] (the first N written), and y must not overlap x
 * (ASR_ERR_ALIAS).  K % 64 == 0, K >= 128 with a norm, and SwiGLU without a
 * norm (else ASR_ERR_UNSUPPORTED).
 * Numerics: the activations enter the tensor cores as two f16 parts (a = hi
 * + lo, both multiplied by the f16 weight), so they keep about 22 bits, and
 * the operand values (x, silu(gate) * up, or (x - x_0) * norm_w and
 * x * norm_w with the norms) must stay below 65504 in magnitude; the
 * sums are fp32 (with the K axis split across CTAs, a residual without a
 * norm adds the parts onto y in an unspecified order, so repeated calls may
 * differ in the last bits).  The norms are folded into the product (the
 * operand is (x - x_0) * norm_w for LayerNorm, x_0 the row's first element,
 * and x * norm_w for RMSNorm; the row statistics and the norm_b terms are
 * applied after the sum), which is the same function up to fp32 rounding.
 * ws: asr_linear_workspace_size(M, N, K) bytes (the largest any norm or input
 * needs), zero-filled before first use and 256-byte aligned (NULL allowed
 * when that size is 0); every call leaves it zero again unless a wait times
 * out (ASR_DEVERR_TIMEOUT), after which it must be zeroed before reuse.  The
 * weight is read before the previous kernel on the stream has finished when
 * that kernel is one of this library's (none of them writes a weight). */
size_t asr_linear_workspace_size(int M, int N, int K);
int asr_linear(const float* x, int64_t x_stride, int norm, const float* norm_w,
               const float* norm_b, float eps, int act, const uint16_t* w, const float* bias,
               int M, int N, int K, int mode, float* y, int64_t y_stride, void* ws,
               size_t ws_bytes, int32_t* dev_err, asr_stream_t stream);

/* Self-attention without a caller workspace (no counterpart in the pages: it
 * is a convenience of this library).  For callers that cannot allocate device
 * memory for a workspace -- a plugin whose host owns every allocation and
 * forbids allocating while it enqueues work, a real-time audio thread that
 * must not wait on an allocator, or a small C program that would rather not
 * size a buffer.  Same arguments, result and errors as asr_self_attn_step,
 * minus ws/ws_bytes: the scratch is a fixed array of
 * asr_noalloc_scratch_bytes() (8 MiB) bytes in device memory, held by every
 * GPU that loads the library until the process exits.  A problem whose
 * workspace (asr_workspace_size(ASR_OP_SELF_ATTN, B, B, 1, heads, head_dim, 0))
 * exceeds it is rejected with ASR_ERR_SCRATCH_LIMIT.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress) with that
 * device current; make that first call before any stream capture.  Each call
 * enqueues a small memset (the counters) and the kernel, and allocates
 * nothing.  All calls on a device share the array: calls that can overlap on
 * the GPU (unordered streams) race and give wrong results.  The address is
 * kept for the life of the process: after cudaDeviceReset on a device that
 * has had a call, this entry point must not be used on it again (the reset
 * unloads the array and the kept address would be stale). */
int asr_self_attn_step_noalloc(const float* q, int64_t q_stride, const uint16_t* cache,
                               int64_t seq_stride, const int32_t* lens, int B, int heads,
                               int head_dim, int capacity, float scale, float* out,
                               int32_t* dev_err, asr_stream_t stream);

/* Size in bytes of the fixed scratch array of asr_self_attn_step_noalloc. */
size_t asr_noalloc_scratch_bytes(void);

/* Workspace bytes needed by an attention entry point on the CURRENT device
 * (its SM count sets the number of key-range pieces).  op: asr_op;
 * n_sources: sequences (self, GQA), groups (cross) or KV heads (prefill);
 * max_beams: 1 except for cross; T: prompt length (prefill only).  Returns 0 for invalid arguments
 * or when no CUDA device is usable. */
size_t asr_workspace_size(int op, int B, int n_sources, int max_beams, int q_heads, int head_dim,
                          int T);

/* Static description of a status code. */
const char* asr_status_string(int status);

/* ABI version (major*100 + minor). */
int asr_version(void);

/* Test support for the bounded waits (no counterpart in the pages).  Arms the
 * next decode-attention launch (asr_self_attn_step, asr_self_attn_append_step,
 * asr_self_attn_reorder_append_step, asr_cross_attn_step, asr_gqa_step or
 * asr_self_attn_step_noalloc) made by
 * the calling host thread: its producer issues no copies, so every pipeline
 * wait of that launch runs out after wait_ns nanoseconds (0 < wait_ns <= 2 s).
 * The kernel then sets ASR_DEVERR_TIMEOUT in dev_err, passes over its
 * remaining work without waiting and returns; its outputs are undefined, the
 * workspace counters are left at zero, and the next call works normally.
 * Nothing faults or hangs.  Returns ASR_OK, or ASR_ERR_INVALID_ARG for a
 * wait_ns out of range (the launch is then not armed). */
int asr_debug_stall_next_decode(uint64_t wait_ns);

/* A promise that lets the decode-attention launches of the calling host
 * thread start earlier (no counterpart in the pages).  Every launch of this
 * library lets the next one on its stream start while it drains, and the
 * next one waits (griddepcontrol.wait) for it to finish before it reads
 * anything.  With ready = 1 the decode-attention entry points
 * (asr_self_attn_step, asr_self_attn_append_step, asr_cross_attn_step,
 * asr_gqa_step, asr_self_attn_step_noalloc) read their lengths (and cross
 * groups), norm weights and cached K/V history before that wait: their
 * producer starts its copies at once and only the queries, the new token,
 * the outputs and the workspace wait.  The caller promises that none of the
 * lengths, groups, norm weights or cached rows a call reads was written by
 * the last few launches before it on the same stream (the one just before
 * it, and one that launch may have let start before its own predecessor
 * finished): true in a steady decode loop (the preceding launches are
 * projections and other layers' attention), false right after a prefill,
 * an append or a beam reorder of the same cache, or an upload of the
 * lengths by a kernel.  A broken promise gives wrong results.  The beam-reorder entry point
 * (asr_self_attn_reorder_append_step) never starts early (it writes a
 * destination cache).  The setting is kept per host thread and is read when
 * a call is made (a captured graph keeps the mode of its capture).  ready:
 * 0 (the default) or 1; ASR_ERR_INVALID_ARG otherwise. */
int asr_set_history_ready(int ready);

#ifdef __cplusplus
}
#endif

#endif /* ASRKV_H */
