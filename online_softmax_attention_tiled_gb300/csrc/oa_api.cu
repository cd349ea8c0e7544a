// oa_api.cu -- the C ABI declared in include/oa.h: host-side validation,
// dispatch to the kernels, the device status word and the wait-limit
// self-test.  Nothing here computes results; every step of the path runs in
// the kernels of this directory.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "oa.h"
#include "oa_internal.h"

namespace {

// Status word written by kernels when a bounded wait expires (site code).
__device__ unsigned int g_status_word;

thread_local char g_last_error[512] = "";
std::atomic<unsigned long long> g_wait_limit_ns{2000000000ull};
constexpr unsigned long long kDefaultLimitNs = 2000000000ull;

oa_status fail(oa_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return s;
}

oa_status ok() {
  g_last_error[0] = '\0';
  return OA_OK;
}

oa_status cuda_fail(cudaError_t e, const char* what) {
  return fail(OA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Device address of the status word for the current device; looked up once
// per device with that device current.
bool status_word(unsigned int** out) {
  constexpr int kMaxDev = 64;
  static unsigned int* cache[kMaxDev] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return false;
  if (cache[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return false;
    cache[dev] = static_cast<unsigned int*>(p);
  }
  *out = cache[dev];
  return true;
}

bool dev_status(oa::DevStatus* st) {
  if (!status_word(&st->word)) return false;
  st->limit_ns = g_wait_limit_ns.load();
  return true;
}

bool aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

constexpr int64_t kMaxGrid = 2147483647;

__global__ void selftest_wait_kernel(oa::DevStatus st) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = oa::smem_addr(&bar);
  if (threadIdx.x == 0) {
    oa::mbar_init(b, 1);
    abort_flag = 0;
    oa::fence_barrier_init();
  }
  __syncthreads();
  // nothing ever arrives on `bar`: the wait must give up after st.limit_ns
  if (threadIdx.x == 0)
    oa::mbar_wait(b, 0, st, reinterpret_cast<volatile int*>(&abort_flag), (oa::K_SELFTEST << 8) | 1);
  __syncthreads();
}

// A debug check whose condition is false: the debug build records the failure and skips the
// store it guards; the release build compiles the check to true and performs the store.
__global__ void selftest_check_kernel(oa::DevStatus st, int* out) {
  if (threadIdx.x == 0 && OA_DCHECK(st, out == nullptr, (oa::K_SELFTEST << 8) | oa::kSiteDebugBase)) *out = 1;
}

}  // namespace

namespace oa {
cudaError_t launch_selftest_check(const DevStatus& st, int* out, cudaStream_t s) {
  selftest_check_kernel<<<1, 32, 0, s>>>(st, out);
  return cudaGetLastError();
}
cudaError_t launch_selftest_wait(const DevStatus& st, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(st);
  return cudaGetLastError();
}
}  // namespace oa

extern "C" {

const char* oa_status_string(int status) {
  switch (status) {
    case OA_OK: return "OA_OK";
    case OA_ERR_INVALID: return "OA_ERR_INVALID: invalid argument";
    case OA_ERR_UNSUPPORTED: return "OA_ERR_UNSUPPORTED: not supported by this build";
    case OA_ERR_CUDA: return "OA_ERR_CUDA: CUDA call failed";
    case OA_ERR_TIMEOUT: return "OA_ERR_TIMEOUT: a bounded device wait expired";
    default: return "unknown oa_status";
  }
}

const char* oa_last_error(void) { return g_last_error; }

int oa_version(void) { return 100; }

void oa_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns == 0 ? kDefaultLimitNs : ns); }

oa_status oa_softmax_rows(const float* x, int64_t rows, int64_t cols, int64_t ld_x, float* y, int64_t ld_y,
                          float* lse, oa_stream_t stream) {
  if (x == nullptr) return fail(OA_ERR_INVALID, "softmax_rows: x is NULL");
  if (rows < 1 || cols < 1) return fail(OA_ERR_INVALID, "softmax_rows: rows and cols must be >= 1");
  if (ld_x < cols) return fail(OA_ERR_INVALID, "softmax_rows: ld_x < cols");
  if (y == nullptr && lse == nullptr) return fail(OA_ERR_INVALID, "softmax_rows: y and lse both NULL");
  if (y != nullptr && ld_y < cols) return fail(OA_ERR_INVALID, "softmax_rows: ld_y < cols");
  if (!aligned(x, 4) || !aligned(y, 4) || !aligned(lse, 4))
    return fail(OA_ERR_INVALID, "softmax_rows: pointers must be 4-byte aligned");
  if (y != nullptr && static_cast<const void*>(y) == static_cast<const void*>(x) && ld_y != ld_x)
    return fail(OA_ERR_INVALID, "softmax_rows: in-place needs ld_y == ld_x");
  if (rows > kMaxGrid / 8) return fail(OA_ERR_INVALID, "softmax_rows: too many rows");
  oa::DevStatus st;
  if (!dev_status(&st)) return fail(OA_ERR_CUDA, "softmax_rows: no current CUDA device");
  cudaError_t e = oa::launch_softmax_rows(x, rows, cols, ld_x, y, ld_y, lse, st, (cudaStream_t)stream);
  return e == cudaSuccess ? ok() : cuda_fail(e, "softmax_rows launch");
}

static oa_status check_attn(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                            int Nk, int d, int causal, float scale, const char* who) {
  if (!q || !k || !v || !o) return fail(OA_ERR_INVALID, "%s: q, k, v and o must be non-NULL", who);
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1) return fail(OA_ERR_INVALID, "%s: sizes must be >= 1", who);
  if (!(std::isfinite(scale) && scale > 0.f)) return fail(OA_ERR_INVALID, "%s: scale must be finite and > 0", who);
  if (causal != 0 && causal != 1) return fail(OA_ERR_INVALID, "%s: causal must be 0 or 1", who);
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return fail(OA_ERR_INVALID, "%s: q/k/v/o must be 16-byte aligned, lse 4-byte", who);
  if ((int64_t)B * H > (int64_t)1 << 30) return fail(OA_ERR_INVALID, "%s: B*H too large", who);
  return OA_OK;
}

static oa_status check_heads(int H, int Hkv, const char* who) {
  if (Hkv < 1 || Hkv > H || H % Hkv != 0)
    return fail(OA_ERR_INVALID, "%s: H_kv must divide H (H %d, H_kv %d)", who, H, Hkv);
  return OA_OK;
}

// Every check of the dense forward, before anything is launched or copied.
static oa_status check_fwd(const void* q, const void* k, const void* v, void* o, float* lse, oa_dtype dt, int B, int H,
                           int Hkv, int Nq, int Nk, int d, int causal, float scale, const int32_t* kv_len,
                           const char* who) {
  oa_status s = check_attn(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale, who);
  if (s != OA_OK) return s;
  if ((s = check_heads(H, Hkv, who)) != OA_OK) return s;
  if (!aligned(kv_len, 4)) return fail(OA_ERR_INVALID, "%s: kv_len must be 4-byte aligned", who);
  if (dt != OA_BF16 && dt != OA_F32) return fail(OA_ERR_INVALID, "%s: unknown dtype %d", who, (int)dt);
  if (dt == OA_BF16 && d != 64 && d != 128)
    return fail(OA_ERR_UNSUPPORTED, "%s: bf16 supports d = 64 or 128 (got %d)", who, d);
  if (dt == OA_F32 && d > 256) return fail(OA_ERR_UNSUPPORTED, "%s: fp32 supports d <= 256 (got %d)", who, d);
  const int64_t grid = (int64_t)B * H * (dt == OA_BF16 ? (Nq + 255) / 256 : (Nq + 15) / 16);
  if (grid > kMaxGrid) return fail(OA_ERR_INVALID, "%s: grid too large", who);
  return OA_OK;
}

// The dense forward on `stream`, arguments already checked.
// qmod > 0: each plane's rows are the queries of several query heads, qmod per head (grouped decode),
// and a row's causal position is its index modulo qmod.
// order_bh / order_sh0: a piece of a call of order_bh planes, from plane order_sh0 (see TcArgs).
static oa_status launch_fwd(const void* q, const void* k, const void* v, void* o, float* lse, oa_dtype dt, int B,
                            int H, int Hkv, int Nq, int Nk, int d, int causal, float scale, const int32_t* kv_len,
                            const oa::DevStatus& st, cudaStream_t stream, const char* who, int qmod = 0,
                            int order_bh = 0, int order_sh0 = 0) {
  if (dt == OA_BF16) {
    oa::TcArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.o = o;
    a.lse = lse;
    a.B = B;
    a.H = H;
    a.Hkv = Hkv;
    a.Nq = Nq;
    a.Nk = Nk;
    a.d = d;
    a.causal = causal;
    a.scale = scale;
    a.kv_len = kv_len;
    a.qmod = qmod;
    a.order_bh = order_bh;
    a.order_sh0 = order_sh0;
    const char* why = nullptr;
    cudaError_t e = oa::launch_attn_tc(a, st, stream, &why);
    if (e != cudaSuccess) return why ? fail(OA_ERR_CUDA, "%s: %s", who, why) : cuda_fail(e, "attn_fwd launch");
    return ok();
  }
  cudaError_t e = oa::launch_attn_f32(static_cast<const float*>(q), static_cast<const float*>(k),
                                      static_cast<const float*>(v), static_cast<float*>(o), lse, B, H, Hkv, Nq, Nk,
                                      d, causal, scale, kv_len, 0, 0, stream);
  return e == cudaSuccess ? ok() : cuda_fail(e, "attn_fwd launch");
}

// Decode with grouped key/value heads (one or a few new tokens per sequence): the g = H / H_kv query
// heads of a group hold g * Nq consecutive rows of q, o and lse, so the batch is also a
// [B, H_kv, g Nq, d] forward in which each plane's K/V rows are streamed once for all the group's
// queries by the tensor-core kernel (0.70 ms instead of 0.97 ms split-KV for B32 H32 H_kv8 Nq1
// Nk32768 d128; 0.35 instead of 1.17 at H_kv 4).  Causal: a row's position is its index modulo Nq.
static bool grouped_queries(oa_dtype dt, int H, int Hkv, int Nq, int d) {
  return dt == OA_BF16 && Hkv < H && (d == 64 || d == 128) && (int64_t)(H / Hkv) * Nq <= 128;
}

static oa_status attn_fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, oa_dtype dt, int B,
                               int H, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                               const int32_t* kv_len, oa_stream_t stream, const char* who) {
  oa_status s = check_fwd(q, k, v, o, lse, dt, B, H, Hkv, Nq, Nk, d, causal, scale, kv_len, who);
  if (s != OA_OK) return s;
  oa::DevStatus st;
  if (!dev_status(&st)) return fail(OA_ERR_CUDA, "%s: no current CUDA device", who);
  // one query is the sequence's last position and sees every key: causal changes nothing
  if (Nq == 1) causal = 0;
  if (grouped_queries(dt, H, Hkv, Nq, d))
    return launch_fwd(q, k, v, o, lse, dt, B, Hkv, Hkv, H / Hkv * Nq, Nk, d, causal, scale, kv_len, st,
                      (cudaStream_t)stream, who, causal ? Nq : 0);
  return launch_fwd(q, k, v, o, lse, dt, B, H, Hkv, Nq, Nk, d, causal, scale, kv_len, st, (cudaStream_t)stream, who);
}

oa_status oa_attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, oa_dtype dt, int B, int H,
                      int Nq, int Nk, int d, int causal, float scale, const int32_t* kv_len, oa_stream_t stream) {
  return attn_fwd_impl(q, k, v, o, lse, dt, B, H, H, Nq, Nk, d, causal, scale, kv_len, stream, "attn_fwd");
}

oa_status oa_attn_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, oa_dtype dt, int B,
                          int H, int H_kv, int Nq, int Nk, int d, int causal, float scale, const int32_t* kv_len,
                          oa_stream_t stream) {
  return attn_fwd_impl(q, k, v, o, lse, dt, B, H, H_kv, Nq, Nk, d, causal, scale, kv_len, stream, "attn_fwd_gqa");
}

// ---------------------------------------------------------------------------
// Host-buffer forward: chunked copies in, kernels, copies out, overlapped on three streams
// the library keeps per device, joined back to the caller's stream.
// ---------------------------------------------------------------------------
namespace {

constexpr int kHostMaxChunks = 64;
constexpr int kHostDefaultChunks = 4;
constexpr int kHostMaxDevices = 64;

struct HostPipe {
  std::mutex mu;  // one call at a time per device: the streams and events are shared
  bool ready = false;
  cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, end = nullptr;
  cudaEvent_t landed[kHostMaxChunks] = {}, done[kHostMaxChunks] = {};
};
HostPipe g_pipes[kHostMaxDevices];

// The device's streams and events, created on first use (with `dev` current).
cudaError_t host_pipe(int dev, HostPipe** out) {
  HostPipe& p = g_pipes[dev];
  if (!p.ready) {
    cudaError_t e = cudaSuccess;
    for (cudaStream_t* st : {&p.in, &p.comp, &p.out})
      if (e == cudaSuccess && *st == nullptr) e = cudaStreamCreateWithFlags(st, cudaStreamNonBlocking);
    for (cudaEvent_t* ev : {&p.start, &p.end})
      if (e == cudaSuccess && *ev == nullptr) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    for (int c = 0; c < kHostMaxChunks && e == cudaSuccess; ++c) {
      if (p.landed[c] == nullptr) e = cudaEventCreateWithFlags(&p.landed[c], cudaEventDisableTiming);
      if (e == cudaSuccess && p.done[c] == nullptr) e = cudaEventCreateWithFlags(&p.done[c], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return e;
    p.ready = true;
  }
  *out = &p;
  return cudaSuccess;
}

size_t round256(size_t n) { return (n + 255) / 256 * 256; }

// First key/value plane of piece c of nch over `units` planes.  The sizes fall linearly (boundaries
// at units (1 - (1 - c / nch)^2), every piece non-empty): what follows the last copy in -- the last
// piece's kernel and copy out -- is then short.  Each piece's kernel costs at least its heaviest item
// (for causal attention, the last query tiles against every key), so a few pieces beat many.
size_t host_piece_bound(int c, int nch, int units) {
  if (c >= nch) return (size_t)units;
  const double t = 1.0 - (double)c / nch;
  const size_t u = (size_t)(units * (1.0 - t * t) + 0.5);
  return std::max((size_t)c, std::min(u, (size_t)(units - (nch - c))));
}

struct HostLayout {
  size_t esize, q, kv, o, lse, total;  // section bytes (each 256-byte aligned), total
};

HostLayout host_layout(oa_dtype dt, int B, int H, int Hkv, int Nq, int Nk, int d) {
  HostLayout L{};
  L.esize = dt == OA_F32 ? 4 : 2;
  L.q = round256((size_t)B * H * Nq * d * L.esize);
  L.kv = round256((size_t)B * Hkv * Nk * d * L.esize);
  L.o = L.q;
  L.lse = round256((size_t)B * H * Nq * 4);
  L.total = L.q + 2 * L.kv + L.o + L.lse;
  return L;
}

}  // namespace

size_t oa_attn_fwd_host_workspace_bytes(oa_dtype dt, int B, int H, int H_kv, int Nq, int Nk, int d) {
  if ((dt != OA_BF16 && dt != OA_F32) || B < 1 || H < 1 || H_kv < 1 || Nq < 1 || Nk < 1 || d < 1) return 0;
  return host_layout(dt, B, H, H_kv, Nq, Nk, d).total;
}

oa_status oa_attn_fwd_host(const void* q_host, const void* k_host, const void* v_host, void* o_host, float* lse_host,
                           oa_dtype dt, int B, int H, int H_kv, int Nq, int Nk, int d, int causal, float scale,
                           int chunks, void* workspace, size_t workspace_bytes, oa_stream_t stream) {
  const char* who = "attn_fwd_host";
  oa_status s = check_fwd(q_host, k_host, v_host, o_host, lse_host, dt, B, H, H_kv, Nq, Nk, d, causal, scale,
                          nullptr, who);
  if (s != OA_OK) return s;
  if (chunks < 0 || chunks > kHostMaxChunks)
    return fail(OA_ERR_INVALID, "%s: chunks must be 0 (default) .. %d", who, kHostMaxChunks);
  const HostLayout L = host_layout(dt, B, H, H_kv, Nq, Nk, d);
  if (workspace == nullptr || workspace_bytes < L.total || !aligned(workspace, 256))
    return fail(OA_ERR_INVALID, "%s: workspace must be 256-byte aligned and >= %zu bytes", who, L.total);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kHostMaxDevices)
    return fail(OA_ERR_CUDA, "%s: no usable current CUDA device", who);
  oa::DevStatus st;
  if (!dev_status(&st)) return fail(OA_ERR_CUDA, "%s: no current CUDA device", who);

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* qd = ws;
  uint8_t* kd = qd + L.q;
  uint8_t* vd = kd + L.kv;
  uint8_t* od = vd + L.kv;
  float* lsed = lse_host ? reinterpret_cast<float*>(od + L.o) : nullptr;
  // chunks over the B * H_kv key/value planes; query planes follow in groups of H / H_kv
  const int units = B * H_kv, g = H / H_kv;
  const int nch = std::min(chunks > 0 ? chunks : kHostDefaultChunks, units);
  const size_t qplane = (size_t)Nq * d * L.esize, kvplane = (size_t)Nk * d * L.esize, lplane = (size_t)Nq * 4;
  const uint8_t* qh = static_cast<const uint8_t*>(q_host);
  const uint8_t* kh = static_cast<const uint8_t*>(k_host);
  const uint8_t* vh = static_cast<const uint8_t*>(v_host);
  uint8_t* oh = static_cast<uint8_t*>(o_host);
  uint8_t* lh = reinterpret_cast<uint8_t*>(lse_host);

  HostPipe* p = nullptr;
  std::lock_guard<std::mutex> lock(g_pipes[dev].mu);
  cudaError_t e = host_pipe(dev, &p);
  if (e != cudaSuccess) return cuda_fail(e, "attn_fwd_host stream set-up");
  const cudaStream_t user = (cudaStream_t)stream;
  // nothing starts before the caller's earlier work on `stream` (which may still use the workspace)
  if ((e = cudaEventRecord(p->start, user)) != cudaSuccess) return cuda_fail(e, "attn_fwd_host record");
  if ((e = cudaStreamWaitEvent(p->in, p->start, 0)) != cudaSuccess) return cuda_fail(e, "attn_fwd_host wait");
  for (int c = 0; c < nch; ++c) {
    const size_t u0 = host_piece_bound(c, nch, units), u1 = host_piece_bound(c + 1, nch, units);
    const size_t nu = u1 - u0;
    // in: this chunk's Q (nu * g planes), K and V (nu planes)
    if ((e = cudaMemcpyAsync(qd + u0 * g * qplane, qh + u0 * g * qplane, nu * g * qplane, cudaMemcpyHostToDevice,
                             p->in)) != cudaSuccess ||
        (e = cudaMemcpyAsync(kd + u0 * kvplane, kh + u0 * kvplane, nu * kvplane, cudaMemcpyHostToDevice, p->in)) !=
            cudaSuccess ||
        (e = cudaMemcpyAsync(vd + u0 * kvplane, vh + u0 * kvplane, nu * kvplane, cudaMemcpyHostToDevice, p->in)) !=
            cudaSuccess ||
        (e = cudaEventRecord(p->landed[c], p->in)) != cudaSuccess)
      return cuda_fail(e, "attn_fwd_host copy in");
    // compute: the chunk as one batch of nu * g query heads over nu key/value heads
    if ((e = cudaStreamWaitEvent(p->comp, p->landed[c], 0)) != cudaSuccess) return cuda_fail(e, "attn_fwd_host wait");
    s = launch_fwd(qd + u0 * g * qplane, kd + u0 * kvplane, vd + u0 * kvplane, od + u0 * g * qplane,
                   lsed ? lsed + u0 * g * Nq : nullptr, dt, 1, (int)(nu * g), (int)nu, Nq, Nk, d, causal, scale,
                   nullptr, st, p->comp, who, 0, B * H, (int)(u0 * g));
    if (s != OA_OK) return s;
    if ((e = cudaEventRecord(p->done[c], p->comp)) != cudaSuccess) return cuda_fail(e, "attn_fwd_host record");
    // out: O and LSE of the chunk
    if ((e = cudaStreamWaitEvent(p->out, p->done[c], 0)) != cudaSuccess) return cuda_fail(e, "attn_fwd_host wait");
    if ((e = cudaMemcpyAsync(oh + u0 * g * qplane, od + u0 * g * qplane, nu * g * qplane, cudaMemcpyDeviceToHost,
                             p->out)) != cudaSuccess)
      return cuda_fail(e, "attn_fwd_host copy out");
    if (lh && (e = cudaMemcpyAsync(lh + u0 * g * lplane, lsed + u0 * g * Nq, nu * g * lplane, cudaMemcpyDeviceToHost,
                                   p->out)) != cudaSuccess)
      return cuda_fail(e, "attn_fwd_host copy out");
  }
  // the caller's stream continues after the last copy out (which follows every chunk's kernel)
  if ((e = cudaEventRecord(p->end, p->out)) != cudaSuccess || (e = cudaStreamWaitEvent(user, p->end, 0)) != cudaSuccess)
    return cuda_fail(e, "attn_fwd_host join");
  return ok();
}

oa_status oa_attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, oa_dtype dt,
                             const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int num_seqs, int H,
                             int H_kv, int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d,
                             int causal, float scale, oa_stream_t stream) {
  const char* who = "attn_fwd_varlen";
  if (!q || !k || !v || !o || !cu_seqlens_q || !cu_seqlens_k)
    return fail(OA_ERR_INVALID, "%s: q, k, v, o and both cu_seqlens must be non-NULL", who);
  if (num_seqs < 1 || H < 1 || d < 1 || total_q < 1 || total_k < 0 || max_seqlen_q < 1 || max_seqlen_k < 0)
    return fail(OA_ERR_INVALID, "%s: need num_seqs, H, d, total_q, max_seqlen_q >= 1 and total_k, max_seqlen_k >= 0",
                who);
  oa_status s = check_heads(H, H_kv, who);
  if (s != OA_OK) return s;
  if (!(std::isfinite(scale) && scale > 0.f)) return fail(OA_ERR_INVALID, "%s: scale must be finite and > 0", who);
  if (causal != 0 && causal != 1) return fail(OA_ERR_INVALID, "%s: causal must be 0 or 1", who);
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4) ||
      !aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4))
    return fail(OA_ERR_INVALID, "%s: q/k/v/o must be 16-byte aligned, lse and cu_seqlens 4-byte", who);
  if (dt != OA_BF16) return fail(OA_ERR_UNSUPPORTED, "%s: bf16 only", who);
  if (d != 64 && d != 128) return fail(OA_ERR_UNSUPPORTED, "%s: d = 64 or 128 (got %d)", who, d);
  if ((int64_t)num_seqs * H * ((max_seqlen_q + 255) / 256) > (int64_t)1 << 31)
    return fail(OA_ERR_INVALID, "%s: too many work items", who);
  oa::DevStatus st;
  if (!dev_status(&st)) return fail(OA_ERR_CUDA, "%s: no current CUDA device", who);
  oa::TcArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.B = num_seqs;
  a.H = H;
  a.Hkv = H_kv;
  a.Nq = max_seqlen_q;
  a.Nk = max_seqlen_k;
  a.d = d;
  a.causal = causal;
  a.scale = scale;
  a.cu_q = cu_seqlens_q;
  a.cu_k = cu_seqlens_k;
  a.Tq = total_q;
  a.Tk = total_k;
  const char* why = nullptr;
  cudaError_t e = oa::launch_attn_tc(a, st, (cudaStream_t)stream, &why);
  if (e != cudaSuccess) return why ? fail(OA_ERR_CUDA, "%s: %s", who, why) : cuda_fail(e, "attn_fwd_varlen launch");
  return ok();
}

oa_status oa_attn_fwd_f32_tiles(const float* q, const float* k, const float* v, float* o, float* lse, int B, int H,
                                int Nq, int Nk, int d, int causal, float scale, const int32_t* kv_len, int Br,
                                int Bc, oa_stream_t stream) {
  oa_status s = check_attn(q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale, "attn_fwd_f32_tiles");
  if (s != OA_OK) return s;
  if (!aligned(kv_len, 4)) return fail(OA_ERR_INVALID, "attn_fwd_f32_tiles: kv_len must be 4-byte aligned");
  if (d > 256) return fail(OA_ERR_UNSUPPORTED, "attn_fwd_f32_tiles: d <= 256");
  if (Br < 1 || Br > 64 || Bc < 1 || Bc > 64) return fail(OA_ERR_INVALID, "attn_fwd_f32_tiles: 1 <= Br, Bc <= 64");
  const size_t smem = sizeof(float) * ((size_t)2 * Br * d + (size_t)2 * Bc * d + (size_t)Br * Bc + 3 * (size_t)Br);
  if (smem > 227 * 1024) return fail(OA_ERR_UNSUPPORTED, "attn_fwd_f32_tiles: tiles need %zu bytes of smem", smem);
  if ((int64_t)B * H * ((Nq + Br - 1) / Br) > kMaxGrid) return fail(OA_ERR_INVALID, "attn_fwd_f32_tiles: grid");
  cudaError_t e =
      oa::launch_attn_f32(q, k, v, o, lse, B, H, H, Nq, Nk, d, causal, scale, kv_len, Br, Bc, (cudaStream_t)stream);
  return e == cudaSuccess ? ok() : cuda_fail(e, "attn_fwd_f32_tiles launch");
}

size_t oa_attn_bwd_workspace_bytes(int B, int H, int Nq, int d) {
  if (B < 1 || H < 1 || Nq < 1 || d < 1) return 0;
  return (oa::attn_bwd_workspace_floats(B, H, Nq, d) * sizeof(float) + 255) / 256 * 256;
}

static oa_status attn_bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dout,
                               const float* lse, void* dq, void* dk, void* dv, oa_dtype dt, int B, int H, int Hkv,
                               int Nq, int Nk, int d, int causal, float scale, void* workspace,
                               size_t workspace_bytes, oa_stream_t stream, const char* who) {
  oa_status s = check_attn(q, k, v, dq, nullptr, B, H, Nq, Nk, d, causal, scale, who);
  if (s != OA_OK) return s;
  if ((s = check_heads(H, Hkv, who)) != OA_OK) return s;
  if (!o || !dout || !lse || !dk || !dv) return fail(OA_ERR_INVALID, "%s: o, dout, lse, dk and dv are required", who);
  if (!aligned(o, 16) || !aligned(dout, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4))
    return fail(OA_ERR_INVALID, "%s: o/dout/dk/dv must be 16-byte aligned, lse 4-byte", who);
  if (dt != OA_BF16) return fail(OA_ERR_UNSUPPORTED, "%s: bf16 only", who);
  if (d != 64 && d != 128) return fail(OA_ERR_UNSUPPORTED, "%s: d = 64 or 128 (got %d)", who, d);
  if ((int64_t)B * Hkv * ((Nk + 127) / 128) > kMaxGrid) return fail(OA_ERR_INVALID, "%s: grid too large", who);
  const size_t need = oa_attn_bwd_workspace_bytes(B, H, Nq, d);
  if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 16))
    return fail(OA_ERR_INVALID, "%s: workspace must be 16-byte aligned and >= %zu bytes", who, need);
  oa::DevStatus st;
  if (!dev_status(&st)) return fail(OA_ERR_CUDA, "%s: no current CUDA device", who);
  oa::BwdArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.B = B;
  a.H = H;
  a.Hkv = Hkv;
  a.Nq = Nq;
  a.Nk = Nk;
  a.d = d;
  a.causal = causal;
  a.scale = scale;
  const char* why = nullptr;
  cudaError_t e = oa::launch_attn_bwd(a, static_cast<float*>(workspace), st, (cudaStream_t)stream, &why);
  if (e != cudaSuccess) return why ? fail(OA_ERR_CUDA, "%s: %s", who, why) : cuda_fail(e, "attn_bwd launch");
  return ok();
}

oa_status oa_attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                      void* dq, void* dk, void* dv, oa_dtype dt, int B, int H, int Nq, int Nk, int d, int causal,
                      float scale, void* workspace, size_t workspace_bytes, oa_stream_t stream) {
  return attn_bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, dt, B, H, H, Nq, Nk, d, causal, scale, workspace,
                       workspace_bytes, stream, "attn_bwd");
}

oa_status oa_attn_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dout,
                          const float* lse, void* dq, void* dk, void* dv, oa_dtype dt, int B, int H, int H_kv, int Nq,
                          int Nk, int d, int causal, float scale, void* workspace, size_t workspace_bytes,
                          oa_stream_t stream) {
  return attn_bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, dt, B, H, H_kv, Nq, Nk, d, causal, scale, workspace,
                       workspace_bytes, stream, "attn_bwd_gqa");
}

oa_status oa_attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dout,
                             const float* lse, void* dq, void* dk, void* dv, oa_dtype dt, const int32_t* cu_seqlens_q,
                             const int32_t* cu_seqlens_k, int num_seqs, int H, int H_kv, int total_q, int total_k,
                             int max_seqlen_q, int max_seqlen_k, int d, int causal, float scale, void* workspace,
                             size_t workspace_bytes, oa_stream_t stream) {
  const char* who = "attn_bwd_varlen";
  oa_status s = check_attn(q, k, v, dq, nullptr, 1, H, total_q, total_k, d, causal, scale, who);
  if (s != OA_OK) return s;
  if ((s = check_heads(H, H_kv, who)) != OA_OK) return s;
  if (!o || !dout || !lse || !dk || !dv || !cu_seqlens_q || !cu_seqlens_k)
    return fail(OA_ERR_INVALID, "%s: o, dout, lse, dk, dv and both cu_seqlens are required", who);
  if (!aligned(o, 16) || !aligned(dout, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4) ||
      !aligned(cu_seqlens_q, 4) || !aligned(cu_seqlens_k, 4))
    return fail(OA_ERR_INVALID, "%s: o/dout/dk/dv must be 16-byte aligned, lse and cu_seqlens 4-byte", who);
  if (num_seqs < 1 || max_seqlen_q < 0 || max_seqlen_k < 1 || max_seqlen_k > total_k)
    return fail(OA_ERR_INVALID, "%s: need num_seqs >= 1 and 1 <= max_seqlen_k <= total_k", who);
  if (dt != OA_BF16) return fail(OA_ERR_UNSUPPORTED, "%s: bf16 only", who);
  if (d != 64 && d != 128) return fail(OA_ERR_UNSUPPORTED, "%s: d = 64 or 128 (got %d)", who, d);
  if ((int64_t)num_seqs * H_kv * ((max_seqlen_k + 127) / 128) > kMaxGrid)
    return fail(OA_ERR_INVALID, "%s: grid too large", who);
  const size_t need = oa_attn_bwd_workspace_bytes(1, H, total_q, d);
  if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 16))
    return fail(OA_ERR_INVALID, "%s: workspace must be 16-byte aligned and >= %zu bytes", who, need);
  oa::DevStatus st;
  if (!dev_status(&st)) return fail(OA_ERR_CUDA, "%s: no current CUDA device", who);
  oa::BwdArgs a{};
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.B = 1;
  a.H = H;
  a.Hkv = H_kv;
  a.Nq = total_q;
  a.Nk = total_k;
  a.d = d;
  a.causal = causal;
  a.scale = scale;
  a.cu_q = cu_seqlens_q;
  a.cu_k = cu_seqlens_k;
  a.num_seqs = num_seqs;
  a.max_seqlen_k = max_seqlen_k;
  const char* why = nullptr;
  cudaError_t e = oa::launch_attn_bwd(a, static_cast<float*>(workspace), st, (cudaStream_t)stream, &why);
  if (e != cudaSuccess) return why ? fail(OA_ERR_CUDA, "%s: %s", who, why) : cuda_fail(e, "attn_bwd_varlen launch");
  return ok();
}

size_t oa_splitkv_workspace_bytes(int B, int H, int Nq, int d, int num_splits) {
  if (B < 1 || H < 1 || Nq < 1 || d < 1 || num_splits < 1) return 0;
  const size_t floats = (size_t)num_splits * (size_t)B * H * Nq * ((size_t)d + 1);
  return (floats * sizeof(float) + 255) / 256 * 256;
}

// Every check of a split-KV call except its scratch memory (shared by oa_attn_splitkv,
// oa_attn_splitkv_gqa and oa_attn_splitkv_static).
static oa_status check_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, oa_dtype dt, int B,
                               int H, int Hkv, int Nq, int Nk, int d, float scale, const int32_t* kv_len,
                               int num_splits, const char* who) {
  oa_status s = check_attn(q, k, v, o, lse, B, H, Nq, Nk, d, 0, scale, who);
  if (s != OA_OK) return s;
  if ((s = check_heads(H, Hkv, who)) != OA_OK) return s;
  if (dt != OA_BF16 && dt != OA_F32) return fail(OA_ERR_INVALID, "%s: unknown dtype %d", who, (int)dt);
  if (!oa::splitkv_supported(dt == OA_BF16, d))
    return fail(OA_ERR_UNSUPPORTED, "%s: unsupported (dtype %d, d %d)", who, (int)dt, d);
  if (num_splits < 1 || num_splits > 1024) return fail(OA_ERR_INVALID, "%s: 1 <= num_splits <= 1024", who);
  if (!aligned(kv_len, 4)) return fail(OA_ERR_INVALID, "%s: kv_len must be 4-byte aligned", who);
  const int64_t R = (int64_t)B * H * Nq;
  if (R * num_splits > kMaxGrid) return fail(OA_ERR_INVALID, "%s: rows * num_splits too large", who);
  return OA_OK;
}

static oa_status attn_splitkv_impl(const void* q, const void* k, const void* v, void* o, float* lse, oa_dtype dt,
                                   int B, int H, int Hkv, int Nq, int Nk, int d, float scale, const int32_t* kv_len,
                                   int num_splits, void* workspace, size_t workspace_bytes, oa_stream_t stream) {
  oa_status s = check_splitkv(q, k, v, o, lse, dt, B, H, Hkv, Nq, Nk, d, scale, kv_len, num_splits, "attn_splitkv");
  if (s != OA_OK) return s;
  const int64_t R = (int64_t)B * H * Nq;
  const size_t need = oa_splitkv_workspace_bytes(B, H, Nq, d, num_splits);
  if (workspace == nullptr || workspace_bytes < need || !aligned(workspace, 16))
    return fail(OA_ERR_INVALID, "attn_splitkv: workspace must be 16-byte aligned and >= %zu bytes", need);
  if (grouped_queries(dt, H, Hkv, Nq, d)) {  // the whole group per plane, no split needed
    oa::DevStatus st;
    if (!dev_status(&st)) return fail(OA_ERR_CUDA, "attn_splitkv: no current CUDA device");
    return launch_fwd(q, k, v, o, lse, dt, B, Hkv, Hkv, H / Hkv * Nq, Nk, d, 0, scale, kv_len, st,
                      (cudaStream_t)stream, "attn_splitkv");
  }
  float* part_o = static_cast<float*>(workspace);
  float* part_lse = part_o + (size_t)num_splits * R * d;
  cudaError_t e = oa::launch_splitkv_partial(q, k, v, dt == OA_BF16, B, H, Hkv, Nq, Nk, d, scale, kv_len, num_splits,
                                             part_o, part_lse, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "attn_splitkv partial launch");
  e = oa::launch_lse_merge(part_o, part_lse, num_splits, R, d, o, dt == OA_BF16, lse, (cudaStream_t)stream);
  return e == cudaSuccess ? ok() : cuda_fail(e, "attn_splitkv merge launch");
}

oa_status oa_attn_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, oa_dtype dt, int B,
                          int H, int Nq, int Nk, int d, float scale, const int32_t* kv_len, int num_splits,
                          void* workspace, size_t workspace_bytes, oa_stream_t stream) {
  return attn_splitkv_impl(q, k, v, o, lse, dt, B, H, H, Nq, Nk, d, scale, kv_len, num_splits, workspace,
                           workspace_bytes, stream);
}

oa_status oa_attn_splitkv_gqa(const void* q, const void* k, const void* v, void* o, float* lse, oa_dtype dt, int B,
                              int H, int H_kv, int Nq, int Nk, int d, float scale, const int32_t* kv_len,
                              int num_splits, void* workspace, size_t workspace_bytes, oa_stream_t stream) {
  return attn_splitkv_impl(q, k, v, o, lse, dt, B, H, H_kv, Nq, Nk, d, scale, kv_len, num_splits, workspace,
                           workspace_bytes, stream);
}

oa_status oa_lse_merge(const float* part_o, const float* part_lse, int S, int64_t R, int d, void* o, oa_dtype o_dt,
                       float* lse, oa_stream_t stream) {
  if (part_lse == nullptr) return fail(OA_ERR_INVALID, "lse_merge: part_lse is NULL");
  if (S < 1 || S > 65535 || R < 1 || d < 0 || d > 1024)
    return fail(OA_ERR_INVALID, "lse_merge: need 1 <= S <= 65535, R >= 1, 0 <= d <= 1024");
  if (d > 0 && (part_o == nullptr || o == nullptr))
    return fail(OA_ERR_INVALID, "lse_merge: part_o and o are required when d > 0");
  if (d == 0 && lse == nullptr) return fail(OA_ERR_INVALID, "lse_merge: nothing to compute (d == 0, lse NULL)");
  if (o_dt != OA_F32 && o_dt != OA_BF16) return fail(OA_ERR_INVALID, "lse_merge: unknown dtype %d", (int)o_dt);
  if (!aligned(part_o, 4) || !aligned(part_lse, 4) || !aligned(lse, 4) || !aligned(o, o_dt == OA_BF16 ? 2 : 4))
    return fail(OA_ERR_INVALID, "lse_merge: misaligned pointer");
  if ((R + 7) / 8 > kMaxGrid) return fail(OA_ERR_INVALID, "lse_merge: R too large");
  cudaError_t e = oa::launch_lse_merge(part_o, part_lse, S, R, d, d > 0 ? o : nullptr, o_dt == OA_BF16, lse,
                                       (cudaStream_t)stream);
  return e == cudaSuccess ? ok() : cuda_fail(e, "lse_merge launch");
}

oa_status oa_sync_status(oa_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "sync_status: stream synchronize");
  unsigned int word = 0;
  e = cudaMemcpyFromSymbol(&word, g_status_word, sizeof word);
  if (e != cudaSuccess) return cuda_fail(e, "sync_status: read status word");
  if (word == 0) return ok();
  const unsigned int zero = 0;
  e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof zero);
  if (e != cudaSuccess) return cuda_fail(e, "sync_status: clear status word");
  if (word == oa::kSiteBadSeqlen)
    return fail(OA_ERR_INVALID, "a packed query sequence is longer than the declared max_seqlen_q; "
                                "its rows past that length were not computed");
  if (word == oa::kSiteBwdBadSeqlen)
    return fail(OA_ERR_INVALID, "a packed key sequence is longer than the declared max_seqlen_k; "
                                "its keys past that length got no dK, dV");
  if ((word & 0xF0u) == oa::kSiteDebugBase)
    return fail(OA_ERR_INVALID, "debug build: bounds or alignment check %u of kernel %u failed (the access was skipped)",
                word & 0x0Fu, word >> 8);
  return fail(OA_ERR_TIMEOUT, "device wait expired: kernel %u, wait site %u", word >> 8, word & 0xFFu);
}

oa_status oa_selftest_debug_check(int* flag, oa_stream_t stream) {
  if (flag == nullptr) return fail(OA_ERR_INVALID, "selftest_debug_check: flag is NULL");
  if (!aligned(flag, 4)) return fail(OA_ERR_INVALID, "selftest_debug_check: flag must be 4-byte aligned");
  oa::DevStatus st;
  if (!dev_status(&st)) return fail(OA_ERR_CUDA, "selftest_debug_check: no current CUDA device");
  cudaError_t e = oa::launch_selftest_check(st, flag, (cudaStream_t)stream);
  return e == cudaSuccess ? ok() : cuda_fail(e, "selftest_debug_check launch");
}

oa_status oa_selftest_wait_timeout(uint64_t limit_ns, oa_stream_t stream) {
  if (limit_ns < 1000ull || limit_ns > 10000000000ull)
    return fail(OA_ERR_INVALID, "selftest_wait_timeout: limit_ns must be in [1e3, 1e10]");
  oa::DevStatus st;
  if (!dev_status(&st)) return fail(OA_ERR_CUDA, "selftest_wait_timeout: no current CUDA device");
  st.limit_ns = limit_ns;
  cudaError_t e = oa::launch_selftest_wait(st, (cudaStream_t)stream);
  return e == cudaSuccess ? ok() : cuda_fail(e, "selftest_wait_timeout launch");
}

}  // extern "C"

// Helpers for entry points defined in other files of the library: record the
// last error / success for oa_last_error(), and fetch the status word.
namespace oa {
oa_status api_fail(oa_status s, const char* msg) { return fail(s, "%s", msg); }
oa_status api_check_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, oa_dtype dt, int B, int H,
                            int Hkv, int Nq, int Nk, int d, float scale, const int32_t* kv_len, int num_splits,
                            const char* who) {
  return check_splitkv(q, k, v, o, lse, dt, B, H, Hkv, Nq, Nk, d, scale, kv_len, num_splits, who);
}
oa_status api_ok() { return ok(); }
bool api_dev_status(DevStatus* st) { return dev_status(st); }
}  // namespace oa
