// noalloc.cu -- a self-attention entry point that needs no caller workspace.
//
// Some callers cannot hand the library a workspace: a plugin whose host owns
// every device allocation and forbids allocating inside its enqueue step, a
// real-time audio thread that must not wait on an allocator (cudaMalloc can
// synchronise the device and takes locks), or a small C program that would
// rather not size and manage a buffer.  For them asr_self_attn_step_noalloc
// runs the ordinary self-attention kernel with its scratch (the split-K
// partial results and the per-sequence counters) in a fixed array that the
// library holds in device memory for the life of the process.
//
// The array is a file-scope __device__ variable, so every GPU that loads this
// library keeps kScratchBytes for it until the process exits.  In host code
// its name is only a host-side stand-in; the device address is obtained once
// per device with cudaGetSymbolAddress (with that device current) and cached.
// Every call on a device shares the array: calls that can overlap on the GPU
// (different streams without ordering) race on it.
#include <mutex>

#include "common.cuh"
#include "decode_attn.cuh"

namespace asrkv {

constexpr size_t kScratchBytes = 8u << 20;  // 8 MiB per device

static __device__ __align__(256) unsigned char g_self_attn_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

// Device address of the scratch array on the current device, looked up once
// per device.  nullptr if the lookup failed.
static void* scratch_address(int* status) {
  static void* addr[kMaxDevices];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    *status = ASR_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_self_attn_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      *status = ASR_ERR_CUDA;
      return nullptr;
    }
    addr[dev] = p;
  }
  *status = ASR_OK;
  return addr[dev];
}

}  // namespace asrkv

using namespace asrkv;

extern "C" size_t asr_noalloc_scratch_bytes(void) { return kScratchBytes; }

extern "C" int asr_self_attn_step_noalloc(const float* q, int64_t q_stride, const uint16_t* cache,
                                          int64_t seq_stride, const int32_t* lens, int B,
                                          int heads, int head_dim, int capacity, float scale,
                                          float* out, int32_t* dev_err, asr_stream_t stream) {
  if (B < 0 || B > ASR_MAX_BATCH || heads < 1 || capacity < 1) return ASR_ERR_INVALID_ARG;
  if ((head_dim != 64 && head_dim != 128) || heads > ASR_MAX_KV_HEADS) return ASR_ERR_UNSUPPORTED;
  if (B == 0) return ASR_OK;
  // the checks asr_self_attn_step makes, done first so that a call that is
  // rejected has enqueued nothing (not even the memset below)
  if (!q || !cache || !lens || !out) return ASR_ERR_INVALID_ARG;
  const int64_t row = 2LL * heads * head_dim;
  if (q_stride < (int64_t)heads * head_dim || seq_stride < (int64_t)capacity * row)
    return ASR_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(cache) || !aligned16(out) || q_stride % 4 != 0 ||
      seq_stride % 8 != 0)
    return ASR_ERR_MISALIGNED;
  if ((int64_t)B * capacity >= (1LL << 31)) return ASR_ERR_UNSUPPORTED;
  const size_t need = asr_workspace_size(ASR_OP_SELF_ATTN, B, B, 1, heads, head_dim, 0);
  if (need == 0) return ASR_ERR_CUDA;
  if (need > kScratchBytes) return ASR_ERR_SCRATCH_LIMIT;
  int st = ASR_OK;
  void* scratch = scratch_address(&st);
  if (!scratch) return st;
  // The kernel expects its per-unit counters (at the start of the workspace)
  // to start at zero.  Each call leaves them at zero, but clear them anyway
  // so that nothing depends on an earlier call having finished normally.
  // This is a memset, not an allocation.
  if (cudaMemsetAsync(scratch, 0, decode_counter_bytes(B, heads), (cudaStream_t)stream) !=
      cudaSuccess)
    return ASR_ERR_CUDA;
  return asr_self_attn_step(q, q_stride, cache, seq_stride, lens, B, heads, head_dim, capacity,
                            scale, out, scratch, kScratchBytes, dev_err, stream);
}
