// abi.cu -- the parts of the C ABI that launch nothing: status strings,
// version, workspace sizing and the per-device SM count.
#include <mutex>

#include "common.cuh"
#include "decode_attn.cuh"
#include "tcgen05.cuh"

namespace asrkv {

int device_sm_count() {
  static int cached[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

cudaError_t ensure_dynamic_smem(const void* fn, int bytes) {
  struct Entry {
    const void* fn;
    int dev, bytes;
  };
  static Entry done[256];
  static int n = 0;
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e;
  }
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (done[i].fn == fn && done[i].dev == dev && done[i].bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e;
  }
  for (int i = 0; i < n; ++i)
    if (done[i].fn == fn && done[i].dev == dev) {
      done[i].bytes = bytes;
      return cudaSuccess;
    }
  if (n < 256) done[n++] = {fn, dev, bytes};
  return cudaSuccess;
}

}  // namespace asrkv

using namespace asrkv;

extern "C" size_t asr_workspace_size(int op, int B, int n_sources, int max_beams, int q_heads,
                                     int head_dim, int T) {
  if (op == ASR_OP_PREFILL_ATTN) {
    // n_sources is the number of KV heads here
    if (B < 1 || B > ASR_MAX_BATCH || T < 1 || n_sources < 1 || n_sources > 16 || q_heads < 1 ||
        q_heads % n_sources != 0 || head_dim != 128)
      return 0;
    return prefill_ws_bytes(B, T, q_heads, n_sources);
  }
  if (op == ASR_OP_MHA_PREFILL || op == ASR_OP_ENCODER_ATTN) {
    if (B < 1 || B > ASR_MAX_BATCH || T < 1 || q_heads < 1 || q_heads > ASR_MAX_KV_HEADS ||
        (head_dim != 64 && head_dim != 128))
      return 0;
    return mha_ws_bytes(B, T, q_heads, head_dim);
  }
  if (B < 0 || n_sources < 1 || n_sources > ASR_MAX_BATCH || max_beams < 1 ||
      max_beams > ASR_MAX_BEAMS || q_heads < 1 || (head_dim != 64 && head_dim != 128))
    return 0;
  switch (op) {
    case ASR_OP_SELF_ATTN:
    case ASR_OP_CROSS_ATTN:
    case ASR_OP_GQA_STEP: {
      const int sms = device_sm_count();
      if (sms <= 0) return 0;
      return decode_ws_bytes(n_sources, op == ASR_OP_CROSS_ATTN ? max_beams : 1, q_heads,
                             head_dim, sms);
    }
    default:
      return 0;
  }
}

extern "C" const char* asr_status_string(int status) {
  switch (status) {
    case ASR_OK: return "ok";
    case ASR_ERR_INVALID_ARG: return "invalid argument";
    case ASR_ERR_UNSUPPORTED: return "unsupported shape";
    case ASR_ERR_MISALIGNED: return "pointer or stride not 16-byte aligned";
    case ASR_ERR_ALIAS: return "source and destination overlap";
    case ASR_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case ASR_ERR_CUDA: return "CUDA error";
    case ASR_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the fixed scratch array";
    default: return "unknown status";
  }
}

extern "C" int asr_version(void) { return 101; }
