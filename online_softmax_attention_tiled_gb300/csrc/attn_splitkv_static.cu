// attn_splitkv_static.cu -- split-KV attention that allocates nothing.
//
// Same computation and kernels as oa_attn_splitkv, but the per-chunk partial
// outputs and LSEs live in a fixed 16 MiB array compiled into this library
// instead of a caller-provided workspace.  It serves callers that cannot
// allocate device memory at the moment they call: code embedded in a host
// application that owns all device memory through its own allocator, or a
// latency-critical path where an allocation could block or fail.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library's module holding it keeps its 16 MiB until the process exits.
// Host code cannot use the array's name as a device address, so the address
// is looked up with cudaGetSymbolAddress once per device (with that device
// current) on the first call there, and then passed to the kernels.  Under
// CUDA's lazy module loading (the default) that first lookup is also what
// loads the module onto the device and commits the 16 MiB, so the first
// call on a device is the one that can fail for lack of device memory or
// wait on the driver; callers should make it once at start-up.
//
// The kernels write every partial they later read (an empty chunk writes
// o_c = 0, lse_c = -inf), so nothing in the array has to start at zero and
// stale contents from an earlier call are never used.  All calls share the
// one array: two calls whose work overlaps on the GPU (different streams, or
// different host threads) race on it and must be serialised by the caller.
#include <mutex>

#include "oa.h"
#include "oa_internal.h"

namespace oa {
oa_status api_fail(oa_status s, const char* msg);
oa_status api_check_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, oa_dtype dt, int B, int H,
                            int Hkv, int Nq, int Nk, int d, float scale, const int32_t* kv_len, int num_splits,
                            const char* who);
oa_status api_ok();
bool api_dev_status(DevStatus* st);
}  // namespace oa

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB
constexpr size_t kScratchFloats = kScratchBytes / sizeof(float);

static __device__ __align__(256) float g_splitkv_scratch[kScratchFloats];

// Device address of g_splitkv_scratch for the current device (nullptr on failure).
float* scratch_address(cudaError_t* err) {
  constexpr int kMaxDev = 64;
  static float* cache[kMaxDev] = {};
  static std::mutex mu;
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDev) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] == nullptr) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_splitkv_scratch);
    if (*err != cudaSuccess) return nullptr;
    cache[dev] = static_cast<float*>(p);
  }
  return cache[dev];
}

}  // namespace

extern "C" oa_status oa_attn_splitkv_static(const void* q, const void* k, const void* v, void* o, float* lse,
                                            oa_dtype dt, int B, int H, int Nq, int Nk, int d, float scale,
                                            const int32_t* kv_len, int num_splits, oa_stream_t stream) {
  using oa::api_fail;
  // the checks of oa_attn_splitkv (one key/value head per query head), then the scratch limit
  const oa_status s =
      oa::api_check_splitkv(q, k, v, o, lse, dt, B, H, H, Nq, Nk, d, scale, kv_len, num_splits, "attn_splitkv_static");
  if (s != OA_OK) return s;
  const int64_t R = (int64_t)B * H * Nq;
  const size_t need = (size_t)num_splits * (size_t)R * ((size_t)d + 1);
  if (need > kScratchFloats)
    return api_fail(OA_ERR_INVALID,
                    "attn_splitkv_static: num_splits*B*H*Nq*(d+1) fp32 partials exceed the 16 MiB static scratch; "
                    "use oa_attn_splitkv with a workspace");
  oa::DevStatus st;
  if (!oa::api_dev_status(&st)) return api_fail(OA_ERR_CUDA, "attn_splitkv_static: no current CUDA device");
  cudaError_t e = cudaSuccess;
  float* part_o = scratch_address(&e);
  if (part_o == nullptr) return api_fail(OA_ERR_CUDA, "attn_splitkv_static: cudaGetSymbolAddress failed");
  float* part_lse = part_o + (size_t)num_splits * R * d;
  e = oa::launch_splitkv_partial(q, k, v, dt == OA_BF16, B, H, H, Nq, Nk, d, scale, kv_len, num_splits, part_o, part_lse,
                                 (cudaStream_t)stream);
  if (e != cudaSuccess) return api_fail(OA_ERR_CUDA, "attn_splitkv_static: partial kernel launch failed");
  e = oa::launch_lse_merge(part_o, part_lse, num_splits, R, d, o, dt == OA_BF16, lse, (cudaStream_t)stream);
  if (e != cudaSuccess) return api_fail(OA_ERR_CUDA, "attn_splitkv_static: merge kernel launch failed");
  return oa::api_ok();
}
