// cross_fill.cu -- the cross-attention K/V of one decoder layer from the
// encoder output, on the 5th-generation tensor cores (next row).
//
// Defines: "wavo 0.1.0, src/whisper/decoder.rs", Decoder::record_cross (a
// GEMM of the encoder rows with the layer's [k | v] weight and a bias
// epilogue, then a pack to f16 cache rows) and Decoder::load (k has no bias,
// v has its own); "Nest whisper-tiny, src/lib.linnet", DecoderLayer.listen.
//
//   cross row t of group g, element n = f16( sum_k enc[g][t][k] * W[n][k]
//                                            + (n >= d ? bias_v[n - d] : 0) )
//
// with K of all heads in elements [0, d) and V in [d, 2d): the cache row
// layout the decode kernels read.  enc and W are f16 (the tensor-core
// operands), the sum is fp32 in tensor memory, the bias is added in fp32 and
// the result rounded to nearest even.
//
// Design: a persistent GEMM, one CTA per SM walking 128 x 256 output tiles
// (tile n fastest, so consecutive CTAs share the A tile through L2; W, at most
// a few MB, stays in L2).  Warp 4 issues TMA loads of A (128 rows x 64 k) and
// B (256 rows of W x 64 k) through a 4-stage ring, warp 5 issues
// tcgen05.mma (M=128, N=256, K=16 each) into one of two TMEM accumulators,
// and warps 0-3 (one thread per output row) drain the other accumulator:
// tcgen05.ld, bias, f16 pack, then through shared memory so that each store
// instruction writes four whole 128-byte row pieces.
#include <mutex>

#include "common.cuh"
#include "tcgen05.cuh"

namespace asrkv {

constexpr int kFillBM = 128, kFillBN = 256, kFillBK = 64;
constexpr int kFillStages = 4;
constexpr int kFillATile = kFillBM * kFillBK * 2;  // 16 KB
constexpr int kFillBTile = kFillBN * kFillBK * 2;  // 32 KB
constexpr int kFillStg = 4 * 32 * 64 * 2;          // output staging: 32 rows x 64 f16 per warp
constexpr int kFillSmem = kFillStages * (kFillATile + kFillBTile) + kFillStg + 1024 + 1024;
constexpr int kFillThreads = 192;  // warps 0-3 epilogue, 4 TMA, 5 MMA

struct FillArgs {
  const float* bias_v;  // [d]
  uint16_t* cross;      // [G][group_stride]
  int64_t group_stride;
  int G, frames, d;
  int m_tiles_per_group, n_tiles, n_tiles_total;
  int32_t* dev_err;
};

__global__ void __launch_bounds__(kFillThreads, 1)
cross_fill_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,
                  const FillArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  unsigned char* sA = smem;                                   // stages x 16 KB
  unsigned char* sB = sA + kFillStages * kFillATile;          // stages x 32 KB
  uint16_t* sStg = reinterpret_cast<uint16_t*>(sB + kFillStages * kFillBTile);  // 4 x 4 KB
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + kFillStages * kFillBTile + kFillStg);
  uint64_t* empty = full + kFillStages;
  uint64_t* acc_full = empty + kFillStages;  // [2]: the accumulator of a tile is complete
  uint64_t* acc_empty = acc_full + 2;        // [2]: the epilogue has read it
  uint64_t* drain = acc_empty + 2;           // every MMA this CTA issued has completed
  uint32_t* tslot = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_any = reinterpret_cast<int*>(tslot + 1);  // some wait of this CTA gave up

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kFillStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    *abort_any = 0;
    fence_barrier_init();
  }
  if (warp == 4) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  grid_launch_dependents();
  grid_dependency_wait();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = *tslot;
  const int k_steps = a.d / kFillBK;
  const int n_tiles_all = a.n_tiles_total;
  bool ok = true;

  int gs = 0;  // ring position (producer: copies issued)
  if (warp == 4) {
    // ======================================================= TMA producer
    for (int tile = blockIdx.x; tile < n_tiles_all && ok; tile += gridDim.x) {
      const int nt = tile % a.n_tiles, mt_all = tile / a.n_tiles;
      const int g = mt_all / a.m_tiles_per_group, mt = mt_all % a.m_tiles_per_group;
      for (int ks = 0; ks < k_steps; ++ks, ++gs) {
        const int s = gs % kFillStages;
        if (gs >= kFillStages && !(ok = mbar_wait_warp(&empty[s], ((gs / kFillStages) - 1) & 1)))
          break;
        mbar_arrive_expect_tx_warp(&full[s], kFillATile + kFillBTile);
        tma_load_3d_warp(sA + s * kFillATile, &ta, ks * kFillBK, mt * kFillBM, g, &full[s]);
        tma_load_3d_warp(sB + s * kFillBTile, &tb, ks * kFillBK, nt * kFillBN, 0, &full[s]);
      }
    }
  } else if (warp == 5) {
    // ======================================================= MMA issuer
    constexpr uint32_t kId = mma_idesc_f16_f32(kFillBM, kFillBN);
    const uint32_t aA = smem_addr(sA), aB = smem_addr(sB);
    int gs = 0, lt = 0;  // ring position, tiles of this CTA so far
    for (int tile = blockIdx.x; tile < n_tiles_all && ok; tile += gridDim.x, ++lt) {
      const int buf = lt & 1;
      // the epilogue must have read this accumulator's previous tile
      if (lt >= 2) ok = mbar_wait_warp(&acc_empty[buf], ((lt >> 1) - 1) & 1);
      tc_fence_after_sync();
      const uint32_t tacc = tbase + 256u * buf;
      for (int ks = 0; ks < k_steps && ok; ++ks, ++gs) {
        const int s = gs % kFillStages;
        ok = mbar_wait_warp(&full[s], (gs / kFillStages) & 1);
        tc_fence_after_sync();
        if (!ok) break;
#pragma unroll
        for (int kk = 0; kk < kFillBK / 16; ++kk)
          mma_f16_warp(tacc, sw128_kmajor_desc(aA + s * kFillATile + kk * 32),
                       sw128_kmajor_desc(aB + s * kFillBTile + kk * 32), kId,
                       (ks > 0 || kk > 0) ? 1u : 0u);
        mma_commit_warp(&empty[s]);  // the stage is free once these finish
      }
      if (ok) mma_commit_warp(&acc_full[buf]);
    }
  } else {
    // ======================================================= epilogue
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    uint16_t* stg = sStg + warp * (32 * 64);
    int lt = 0;
    for (int tile = blockIdx.x; tile < n_tiles_all && ok; tile += gridDim.x, ++lt) {
      const int buf = lt & 1;
      const int nt = tile % a.n_tiles, mt_all = tile / a.n_tiles;
      const int g = mt_all / a.m_tiles_per_group, mt = mt_all % a.m_tiles_per_group;
      ok = mbar_wait_warp(&acc_full[buf], (lt >> 1) & 1);
      if (!ok) break;
      tc_fence_after_sync();
      const uint32_t tacc = tbase + 256u * buf + lane_off;
      const int r0 = mt * kFillBM + warp * 32;  // frame of lane 0's row
      uint16_t* gbase = a.cross + (int64_t)g * a.group_stride;
#pragma unroll 1
      for (int c = 0; c < kFillBN / 64; ++c) {
        float v[64];
        tmem_ld32(tacc + c * 64, v);
        tmem_ld32(tacc + c * 64 + 32, v + 32);
        tmem_wait_ld();
        const int n0 = nt * kFillBN + c * 64;  // first output column of the chunk
        if (n0 >= a.d) {  // V columns carry the bias (chunks never straddle d)
          const float4* bp = reinterpret_cast<const float4*>(a.bias_v + (n0 - a.d));
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float4 bv = __ldg(bp + e);
            v[4 * e] += bv.x;
            v[4 * e + 1] += bv.y;
            v[4 * e + 2] += bv.z;
            v[4 * e + 3] += bv.w;
          }
        }
        // row `lane` of the warp: 64 f16 = eight 16-byte chunks, chunk q at
        // q ^ (lane % 8)
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          uint4 u;
          __half2* h = reinterpret_cast<__half2*>(&u);
#pragma unroll
          for (int e = 0; e < 4; ++e) h[e] = __floats2half2_rn(v[8 * q + 2 * e], v[8 * q + 2 * e + 1]);
          *reinterpret_cast<uint4*>(stg + lane * 64 + ((q ^ (lane & 7)) * 8)) = u;
        }
        __syncwarp();
        // each instruction: four rows x 128 bytes
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          const int rr = it * 4 + (lane >> 3), q = lane & 7;
          const uint4 u = *reinterpret_cast<const uint4*>(stg + rr * 64 + ((q ^ (rr & 7)) * 8));
          const int t = r0 + rr;
          if (t < a.frames)
            *reinterpret_cast<uint4*>(gbase + (int64_t)t * 2 * a.d + n0 + q * 8) = u;
        }
        __syncwarp();
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
  }
  if (!ok && lane == 0) {
    set_dev_err(a.dev_err, ASR_DEVERR_TIMEOUT);
    atomicExch(abort_any, 1);
  }
  tc_fence_before_sync();
  __syncthreads();
  // After a wait gave up, nothing may still be in flight into this CTA's
  // shared memory or tensor memory when it frees them and leaves: the
  // producer waits (bounded) for the copies it issued (only the last ring's
  // worth can be pending), the MMA warp for every MMA it issued (a commit
  // tracks all of them).
  if (*reinterpret_cast<volatile int*>(abort_any)) {
    if (warp == 4) {
      for (int i = max(0, gs - kFillStages); i < gs; ++i)
        mbar_wait_warp(&full[i % kFillStages], (i / kFillStages) & 1);
    } else if (warp == 5) {
      mma_commit_warp(drain);
      mbar_wait_warp(drain, 0);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after_sync();
    tmem_dealloc(tbase, 512);
  }
}

}  // namespace asrkv

using namespace asrkv;

extern "C" int asr_cross_kv_fill(const uint16_t* enc, const uint16_t* w, const float* bias_v,
                                 int G, int frames, int d, uint16_t* cross, int64_t group_stride,
                                 int32_t* dev_err, asr_stream_t stream) {
  if (G < 0 || G > ASR_MAX_BATCH || frames < 1 || d < 1) return ASR_ERR_INVALID_ARG;
  if (d % 128 != 0 || d > 8192) return ASR_ERR_UNSUPPORTED;
  if (G == 0) return ASR_OK;
  if (!enc || !w || !bias_v || !cross) return ASR_ERR_INVALID_ARG;
  if (group_stride < (int64_t)frames * 2 * d) return ASR_ERR_INVALID_ARG;
  if (!aligned16(enc) || !aligned16(w) || !aligned16(bias_v) || !aligned16(cross) ||
      group_stride % 8 != 0)
    return ASR_ERR_MISALIGNED;
  if (ensure_dynamic_smem((const void*)cross_fill_kernel, kFillSmem) != cudaSuccess)
    return ASR_ERR_CUDA;
  // A: enc (dims d, frames, G); B: W (dims d, 2d)
  CUtensorMap ta, tb;
  if (!make_tmap_f16_3d(&ta, enc, d, frames, G, (uint64_t)d * 2, (uint64_t)frames * d * 2, kFillBK,
                        kFillBM) ||
      !make_tmap_f16_3d(&tb, w, d, 2 * (uint64_t)d, 1, (uint64_t)d * 2, (uint64_t)2 * d * d * 2,
                        kFillBK, kFillBN))
    return ASR_ERR_CUDA;
  FillArgs fa = {};
  fa.bias_v = bias_v;
  fa.cross = cross;
  fa.group_stride = group_stride;
  fa.G = G;
  fa.frames = frames;
  fa.d = d;
  fa.m_tiles_per_group = (frames + kFillBM - 1) / kFillBM;
  fa.n_tiles = 2 * d / kFillBN;
  fa.n_tiles_total = G * fa.m_tiles_per_group * fa.n_tiles;
  fa.dev_err = dev_err;
  const int sms = device_sm_count();
  if (sms <= 0) return ASR_ERR_CUDA;
  const int ctas = fa.n_tiles_total < sms ? fa.n_tiles_total : sms;
  cudaError_t e = launch_pdl(cross_fill_kernel, dim3(ctas), dim3(kFillThreads), (size_t)kFillSmem,
                             (cudaStream_t)stream, ta, tb, fa);
  return e == cudaSuccess ? ASR_OK : ASR_ERR_CUDA;
}
