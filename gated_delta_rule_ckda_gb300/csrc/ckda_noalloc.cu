// ckda_noalloc.cu -- the forward for callers that must not allocate device
// memory.
//
// ckda_fwd takes a caller-owned workspace: a status word plus, for packed
// sequences, the longest-first work order.  Some callers cannot provide one.
// Examples are a host application whose device memory is carved up once at
// start-up (cudaMalloc is forbidden afterwards), or a plugin whose host owns
// the only allocator and exposes no handle to it.  This variant keeps that
// scratch in a fixed array in this library's device memory instead, and then
// runs exactly the ckda_fwd path.
#include "ckda_internal.cuh"

#include <cuda.h>
#include <mutex>

namespace ckda {
namespace {

constexpr int kNoAllocMaxSeqs = 65536;
constexpr size_t kNoAllocBytes = kWsStatusBytes + (size_t)kNoAllocMaxSeqs * sizeof(int32_t);

// Every GPU that loads this library holds this array (256 KiB + 256 B) until
// the process exits.  In host code the name is only a stand-in: the device
// address comes from cudaGetSymbolAddress, per context.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

// The address of a __device__ array belongs to the CUDA context that loaded
// this module, not to the device index: a plugin host may make its own
// driver-API context current, and cudaDeviceReset makes the runtime load the
// module again in a fresh primary context.  So the set-up is done once per
// context, keyed by the context's unique id (cuCtxGetId), and its result is
// never reused in another context.
using PFN_ctx_get_current = CUresult (*)(CUcontext*);
using PFN_ctx_get_id = CUresult (*)(CUcontext, unsigned long long*);

struct DriverFns {
  PFN_ctx_get_current get_current = nullptr;
  PFN_ctx_get_id get_id = nullptr;
};
const DriverFns& driver_fns() {
  static DriverFns f;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<PFN_ctx_get_current>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      f.get_id = reinterpret_cast<PFN_ctx_get_id>(p);
  });
  return f;
}

constexpr int kCacheSlots = 64;
std::mutex g_mu;
unsigned long long g_ctx_id[kCacheSlots] = {};
void* g_scratch_addr[kCacheSlots] = {};
int g_used = 0;

// Device address of the scratch array in the current context (set up on the
// first call in that context).
ckda_status scratch_for_current_context(void** out) {
  void* p = nullptr;
  const DriverFns& f = driver_fns();
  unsigned long long id = 0;
  bool keyed = false;
  if (f.get_current && f.get_id) {
    CUcontext ctx = nullptr;
    if (f.get_current(&ctx) == CUDA_SUCCESS && ctx && f.get_id(ctx, &id) == CUDA_SUCCESS)
      keyed = true;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (keyed) {
    for (int i = 0; i < g_used; ++i)
      if (g_ctx_id[i] == id) {
        *out = g_scratch_addr[i];
        return CKDA_OK;
      }
  }
  // no context yet (the runtime creates the primary one here), no cached
  // entry, or no way to identify the context: look the address up now
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return CKDA_ERR_CUDA;
  if (keyed && g_used < kCacheSlots) {
    g_ctx_id[g_used] = id;
    g_scratch_addr[g_used] = p;
    ++g_used;
  }
  *out = p;
  return CKDA_OK;
}

}  // namespace
}  // namespace ckda

extern "C" ckda_status ckda_fwd_noalloc(const void* q, const void* k, const void* v,
                                        const void* alpha, const void* beta, const float* h0,
                                        void* o, float* hT, const int32_t* cu_seqlens,
                                        int num_seqs, int B, int H, int T, int dk, int dv,
                                        ckda_dtype io_dtype, float scale, int chunk_size,
                                        void* stream) {
  using namespace ckda;
  if (cu_seqlens && num_seqs > kNoAllocMaxSeqs) return CKDA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const ckda_status st = scratch_for_current_context(&scratch);
  if (st != CKDA_OK) return st;
  return ckda_fwd(q, k, v, alpha, beta, h0, o, hT, cu_seqlens, num_seqs, B, H, T, dk, dv,
                  io_dtype, scale, chunk_size, scratch, kNoAllocBytes, stream);
}
