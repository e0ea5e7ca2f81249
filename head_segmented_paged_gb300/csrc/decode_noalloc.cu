// Decode attention for callers that cannot allocate device memory per call:
// serving runtimes that forbid cudaMalloc on the request path, or code that
// runs where a caller-sized workspace cannot be obtained. The split-KV
// partials live in a fixed device array defined in this file instead of a
// caller workspace; everything else is the regular decode path. The paper
// has no counterpart: this is a packaging choice of this library.
#include <cstdio>
#include <mutex>

#include "../../include/segkv.h"
#include "segkv_internal.h"

struct segkv;

namespace skv {
size_t decode_partials_bytes(segkv* h, int layer, const int32_t* seq_lens,
                             const int32_t* seq_ids, int n);
int set_error(segkv* h, int code, const char* msg);
int handle_device(const segkv* h);
}  // namespace skv

namespace {

// The scratch: held by every GPU that loads this library until the process
// exits. Each call overwrites it; calls that overlap on the GPU race.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SEGKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device (host code may not use
// the array's name as an address). Looked up once per device.
cudaError_t scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int segkv_decode_attn_noalloc(segkv_t h, int layer, const void* q,
                                         const int32_t* seq_lens, const int32_t* seq_ids, int n,
                                         void* o, segkv_stream_t stream) {
  if (!h) return SEGKV_ERR_INVALID_ARG;
  const int hdev = skv::handle_device(h);
  if (hdev < 0) return skv::set_error(h, SEGKV_ERR_INVALID_ARG, "host-only handle has no pools");
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return skv::set_error(h, SEGKV_ERR_CUDA, cudaGetErrorString(e));
  if (dev != hdev || dev >= kMaxDevices)
    return skv::set_error(h, SEGKV_ERR_INVALID_ARG,
                          "the handle's device must be current for the no-alloc decode call");
  const size_t need = skv::decode_partials_bytes(h, layer, seq_lens, seq_ids, n);
  if (need > SEGKV_NOALLOC_SCRATCH_BYTES) {
    char msg[256];
    std::snprintf(msg, sizeof msg,
                  "this decode needs %zu bytes of partials; the no-alloc entry point holds at "
                  "most %zu (use segkv_decode_attn with a workspace)",
                  need, static_cast<size_t>(SEGKV_NOALLOC_SCRATCH_BYTES));
    return skv::set_error(h, SEGKV_ERR_INVALID_ARG, msg);
  }
  void* scratch = nullptr;
  e = scratch_address(dev, &scratch);
  if (e != cudaSuccess) return skv::set_error(h, SEGKV_ERR_CUDA, cudaGetErrorString(e));
  // The partials need no clearing: every split unit writes its whole slot
  // before the combine pass reads it.
  return segkv_decode_attn(h, layer, q, seq_lens, seq_ids, n, o, scratch,
                           SEGKV_NOALLOC_SCRATCH_BYTES, stream);
}
