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

#include <mutex>

namespace ckda {
namespace {

constexpr int kNoAllocMaxSeqs = 65536;
constexpr size_t kNoAllocBytes = kWsStatusBytes + (size_t)kNoAllocMaxSeqs * sizeof(int32_t);

// Every GPU that loads this library holds this array (256 KiB + 256 B) until
// the process exits.  In host code the name is only a stand-in: the device
// address comes from cudaGetSymbolAddress, per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up on the
// first call for that device).
ckda_status scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return CKDA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return CKDA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return CKDA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
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
  const ckda_status st = scratch_for_current_device(&scratch);
  if (st != CKDA_OK) return st;
  return ckda_fwd(q, k, v, alpha, beta, h0, o, hT, cu_seqlens, num_seqs, B, H, T, dk, dv,
                  io_dtype, scale, chunk_size, scratch, kNoAllocBytes, stream);
}
