// paged_decode_attention_noalloc: the split-K decode with its scratch in a
// fixed device array that ships with this library, for callers that may not
// allocate device memory at call time.
//
// Who needs it: a caller whose device memory is already spoken for when it
// runs decode -- for example a serving runtime that handed all free memory to
// its KV pool at start-up and forbids any later allocation, or a plugin host
// whose calling convention has no workspace argument and whose code must not
// call cudaMalloc (a synchronising call that can also fail mid-serving).
// Such a caller passes only inputs and outputs; the split-K partial results
// go to the static array below instead of a caller workspace.
//
// What it costs: every GPU that loads this library reserves
// PAGED_DECODE_STATIC_SCRATCH_BYTES for the array until the process exits.

#include <mutex>

#include "common.cuh"
#include "internal.h"

// Split-K partial outputs and (max, sum) pairs of one call.  Shared by every
// call on a device; it keeps the last call's contents.  Nothing in it needs
// to start at zero: the decode kernel writes every partial that the reduce
// kernel then reads, within the same call.
static __device__ __align__(256) unsigned char g_decode_scratch[PAGED_DECODE_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 256;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};  // context the address belongs to

// Unique id of the calling thread's current CUDA context (cuCtxGetId, reached
// through the runtime's driver entry point).  False when it cannot be told.
// Called with g_scratch_mutex held.
bool current_context_id(unsigned long long* id) {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static bool looked_up = false;
  if (!looked_up) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(f);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(f);
    looked_up = true;
  }
  CUcontext ctx = nullptr;
  return get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx &&
         get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of g_decode_scratch on `device`, which must be current.  In
// host code the symbol is only a host-side stand-in, so a kernel must be given
// this address, never the symbol itself.  The address is looked up once per
// device and context: if the device's context was destroyed and made again
// (cudaDeviceReset), the module is loaded anew and the address is looked up
// again; if the context cannot be identified it is looked up on every call.
cudaError_t scratch_address(int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  unsigned long long ctx = 0;
  const bool known = current_context_id(&ctx);
  if (!g_scratch_addr[device] || !known || g_scratch_ctx[device] != ctx) {
    void* addr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&addr, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[device] = addr;
    g_scratch_ctx[device] = known ? ctx : 0;
  }
  *out = g_scratch_addr[device];
  return cudaSuccess;
}

}  // namespace

extern "C" kv_status paged_decode_attention_noalloc(
    kv_pool* pool, const void* q, int32_t n_q_heads, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t batch,
    int32_t max_context_len, float scale, int32_t sliding_window, float* out, void* stream) {
  if (!pool || batch < 0 || n_q_heads <= 0 || max_context_len < 0) return KV_ERR_INVALID_ARG;
  // The same partitioning as paged_decode_attention, so both give the same
  // result; refuse sizes whose partials would not fit the fixed array.
  const pkv::DecodePlan plan =
      pkv::plan_decode(pool, batch, n_q_heads, max_context_len, sliding_window);
  if (plan.workspace_bytes > PAGED_DECODE_STATIC_SCRATCH_BYTES) return KV_ERR_INVALID_ARG;

  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) {
    cudaGetLastError();
    return KV_ERR_CUDA;
  }
  if (prev != pool->device && cudaSetDevice(pool->device) != cudaSuccess) {
    cudaGetLastError();
    return KV_ERR_CUDA;
  }
  void* scratch = nullptr;
  const cudaError_t e = scratch_address(pool->device, &scratch);
  if (prev != pool->device) cudaSetDevice(prev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return KV_ERR_CUDA;
  }
  return paged_decode_attention(pool, q, n_q_heads, block_tables, max_blocks_per_seq,
                                context_lens, batch, max_context_len, scale, sliding_window, out,
                                scratch, PAGED_DECODE_STATIC_SCRATCH_BYTES, stream);
}
