// Decode attention for callers that cannot give this library any scratch
// memory.
//
// tq_decode_attention needs a workspace (per-step query fragments and the
// split-context partial results), which its caller allocates.  Some callers
// cannot do that: a plugin running inside a host framework that owns all
// device memory and forbids extra allocations by third-party code, or a
// latency-critical loop that must not call cudaMalloc (it can synchronise the
// device) and has no memory pool to draw from.  tq_decode_attention_static
// serves them: its scratch is one array compiled into this library, so the
// call itself allocates nothing.
//
// Cost and limits of that choice:
//   * the array is kStaticScratchBytes (4 MiB) and every GPU that loads the
//     library reserves it until the process exits;
//   * a call whose workspace would exceed it is rejected with TQ_EINVAL and
//     an error message, before anything is launched;
//   * all calls share the one array and it keeps whatever the last call left
//     there; nothing in it has to start at zero, because each call writes all
//     the scratch it later reads.  Calls whose work overlaps on the GPU (for
//     example on two streams) race on the array: serialise them.
//   * host code cannot use the array's name as a device address (on the host
//     it only names a stand-in object), so the first call on each device
//     looks up the address with cudaGetSymbolAddress while that device is
//     current and remembers it.  Make that first call before any stream
//     capture.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "tq.h"
#include "tq_internal.cuh"

namespace tq {
tq_status report_error(tq_status st, const char* msg);
}

namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_attn_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_attn_scratch on the current device (looked up once per device).
tq_status scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return tq::report_error(TQ_ECUDA, "tq_decode_attention_static: no current CUDA device");
  if (dev < 0 || dev >= kMaxDevices)
    return tq::report_error(TQ_EUNSUPPORTED, "tq_decode_attention_static: device index out of range");
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_scratch);
    if (e != cudaSuccess || !p) {
      char msg[256];
      snprintf(msg, sizeof(msg), "tq_decode_attention_static: cudaGetSymbolAddress failed: %s",
               cudaGetErrorString(e));
      return tq::report_error(TQ_ECUDA, msg);
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return TQ_OK;
}

}  // namespace

extern "C" tq_status tq_decode_attention_static(const tq_codebook* kcb, const tq_codebook* vcb, const void* kcache,
                                                const void* vcache, int32_t B, int32_t Hq, int32_t Hkv,
                                                int64_t capacity, const int32_t* seq_lens, const float* q,
                                                float scale, float* out, void* stream) {
  const tq::NvtxRange nvtx_range("tq_decode_attention_static");
  if (!kcb || !vcb) return tq::report_error(TQ_EINVAL, "tq_decode_attention_static: codebook is NULL");
  const size_t need = tq_decode_attention_workspace(kcb, B, Hq, Hkv, capacity);
  if (need > kStaticScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "tq_decode_attention_static: this call needs %zu bytes of scratch but the built-in array holds %zu; "
             "use tq_decode_attention with a workspace",
             need, kStaticScratchBytes);
    return tq::report_error(TQ_EINVAL, msg);
  }
  void* scratch = nullptr;
  const tq_status st = scratch_address(&scratch);
  if (st != TQ_OK) return st;
  return tq_decode_attention(kcb, vcb, kcache, vcache, B, Hq, Hkv, capacity, seq_lens, q, scale, out, scratch,
                             kStaticScratchBytes, stream);
}
