// softmax_rows.cu -- bandwidth-bound row softmax with per-row log-sum-exp.
//
// One read of x per element when the row fits on chip (the common case):
//   1. each thread keeps its E elements in registers and forms its own
//      (m, l): m = max, l = sum exp(x - m)  (tile recurrence of the
//      roadmap page s.4, with the thread's elements as the tile);
//   2. the (m, l) pairs are merged with warp shuffles, then across the
//      CTA's warps, then across the CTAs of a thread-block cluster through
//      distributed shared memory (interview lesson Step 1: the merge is
//      associative and commutative, so any tree works);
//   3. y = exp(x - m) / l is written from the registers.
// Loads and stores are 128-bit and coalesced when the rows are 16-byte
// aligned.  Up to 65,536 columns a row is held on chip: 8192 columns per
// CTA (256 threads x 32 fp32 in registers), up to 8 CTAs of a cluster per
// row.  Wider rows give each CTA a slice of two such pieces (16,384
// columns), up to 16 CTAs of a cluster per row where the device schedules
// that non-portable size, and the CTA reads its slice in a statistics pass,
// then writes the output of the piece still in its registers and reads the
// others again: the second read of a 64 KB slice, issued right after the
// first, comes back from L2, so X still crosses HBM once.  This
// measured faster than holding 16,384 columns a CTA in registers (two CTAs
// per SM: 3.4 against 4.9 TB/s at 256 x 262,144) and than one-read clusters
// of 16 x 8192 (4.5 against 5.3 TB/s at 512 x 131,072).
// A row whose elements are all -inf has l = 0: it writes y = +0.0 and
// lse = -inf without forming -inf - -inf anywhere.
#include <cooperative_groups.h>

#include "oa_internal.h"

namespace oa {
namespace {

constexpr int kMaxThreads = 256;

struct ML {
  float m, l;
};

// (m, l) merge with 0 as the reference when both maxima are -inf.
__device__ __forceinline__ ML ml_merge(ML a, ML b) {
  const float m = fmaxf(a.m, b.m);
  const float ref = (m == -INFINITY) ? 0.f : m;
  return {m, a.l * expf(a.m - ref) + b.l * expf(b.m - ref)};
}

__device__ __forceinline__ ML warp_merge(ML v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    ML o{__shfl_xor_sync(0xffffffffu, v.m, off), __shfl_xor_sync(0xffffffffu, v.l, off)};
    v = ml_merge(v, o);
  }
  return v;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Split exit barrier: arrive (no release: it orders nothing but the peers'
// finished reads of this CTA's shared memory) as soon as the remote reads are
// done, wait just before exiting -- so no CTA waits for its output stores.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }
__device__ __forceinline__ float ld_dsmem_f32(uint32_t local_addr, uint32_t rank) {
  uint32_t remote;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

// Loads the E elements this thread owns in the piece starting at column
// `base` (relative to the row), -inf outside [.., end).  VEC: groups of four
// consecutive columns, group g at base + (g*T + t)*4.  Scalar: column
// base + i*T + t.
template <int E, bool VEC, bool STREAM>
__device__ __forceinline__ void load_piece(const float* __restrict__ xr, int64_t base, int64_t end, float (&v)[E]) {
  const int T = blockDim.x, t = threadIdx.x;
  if constexpr (VEC) {
#pragma unroll
    for (int g = 0; g < E / 4; ++g) {
      const int64_t c = base + ((int64_t)g * T + t) * 4;
      if (c + 3 < end) {
        const float4 f = STREAM ? __ldcs(reinterpret_cast<const float4*>(xr + c))
                                : __ldg(reinterpret_cast<const float4*>(xr + c));
        v[4 * g] = f.x, v[4 * g + 1] = f.y, v[4 * g + 2] = f.z, v[4 * g + 3] = f.w;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) v[4 * g + e] = (c + e < end) ? xr[c + e] : -INFINITY;
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const int64_t c = base + (int64_t)i * T + t;
      v[i] = (c < end) ? (STREAM ? __ldcs(xr + c) : __ldg(xr + c)) : -INFINITY;
    }
  }
}

template <int E>
__device__ __forceinline__ ML thread_stats(const float (&v)[E]) {
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < E; ++i) m = fmaxf(m, v[i]);
  if (m == -INFINITY) return {m, 0.f};
  float l0 = 0.f, l1 = 0.f;
#pragma unroll
  for (int i = 0; i < E; i += 2) {
    l0 += ex2((v[i] - m) * kLog2e);
    if (i + 1 < E) l1 += ex2((v[i + 1] - m) * kLog2e);
  }
  return {m, l0 + l1};
}

// exp(x - m) / l.  Relative error bound for every output that is a normal
// fp32 number (x - m > -87.4): rounding x - m costs |x - m| * 2^-24 <= 5.2e-6,
// expf ~1 ulp, the product with 1/l two roundings, and l itself (a sum of
// terms <= 1 with one dominant 1) carries ~1e-6 -- together under 1e-5.
// `ref` is the row max, or 0 for a row that is entirely -inf (then 1/l is 0):
// x = -inf gives exp(-inf) = +0.0 exactly and -inf - -inf never forms.
__device__ __forceinline__ float softmax_value(float x, float ref, float inv_l) { return expf(x - ref) * inv_l; }

template <int E, bool VEC>
__device__ __forceinline__ void store_piece(float* __restrict__ yr, int64_t base, int64_t end, const float (&v)[E],
                                            float ref, float inv_l) {
  const int T = blockDim.x, t = threadIdx.x;
  if constexpr (VEC) {
#pragma unroll
    for (int g = 0; g < E / 4; ++g) {
      const int64_t c = base + ((int64_t)g * T + t) * 4;
      if (c + 3 < end) {
        float4 f;
        f.x = softmax_value(v[4 * g], ref, inv_l);
        f.y = softmax_value(v[4 * g + 1], ref, inv_l);
        f.z = softmax_value(v[4 * g + 2], ref, inv_l);
        f.w = softmax_value(v[4 * g + 3], ref, inv_l);
        __stcs(reinterpret_cast<float4*>(yr + c), f);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (c + e < end) yr[c + e] = softmax_value(v[4 * g + e], ref, inv_l);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const int64_t c = base + (int64_t)i * T + t;
      if (c < end) __stcs(yr + c, softmax_value(v[i], ref, inv_l));
    }
  }
}

// CTAs per SM the register budget is cut for: five 256-thread CTAs (48 registers) hide each
// other's load and reduction phases better than four (64 registers: 0.194 -> 0.187 ms at
// 4096 x 32768; three at 80 registers were 0.8 % slower than four); the scalar 32-element
// instance runs three (at four, 64 registers, its streaming branch spills).
template <int E, bool VEC>
constexpr int kSoftmaxMinBlocks = (E == 32 && !VEC) ? 3 : 5;

// grid.x = rows * cluster; the `cluster` CTAs of a row split its columns into
// slices of `slice` columns (a multiple of 4).  PAR: the cluster merge reads the peers'
// statistics in parallel (the instance for clusters of more than 4 CTAs).
template <int E, bool VEC, bool PAR = false>
__global__ void __launch_bounds__(kMaxThreads, kSoftmaxMinBlocks<E, VEC>)
    softmax_rows_kernel(const float* __restrict__ x, int64_t rows, int64_t cols, int64_t ld_x, float* __restrict__ y,
                        int64_t ld_y, float* __restrict__ lse, int cluster, int64_t slice, DevStatus status) {
  __shared__ ML warp_ml[kMaxThreads / 32];
  __shared__ ML cta_ml;  // this CTA's merged statistics (read by peers)
  __shared__ ML row_ml;  // statistics of the whole row

  const int T = blockDim.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t rank = (cluster > 1) ? cluster_rank() : 0u;
  const int64_t row = blockIdx.x / cluster;
  const float* xr = x + row * ld_x;
  const int64_t c0 = (int64_t)rank * slice;
  // (debug build) a row past the tensor or a vector path on unaligned memory leaves the slice
  // empty -- no loads or stores -- while the CTA still takes part in the cluster's barriers
  const bool in_ok =
      OA_DCHECK(status, row < rows, (K_SOFTMAX << 8) | kSiteDebugBase) &&
      (!VEC || OA_DCHECK(status, (reinterpret_cast<uintptr_t>(xr + c0) & 15) == 0 &&
                                 (y == nullptr || (reinterpret_cast<uintptr_t>(y + row * ld_y + c0) & 15) == 0),
                         (K_SOFTMAX << 8) | (kSiteDebugBase + 1)));
  const int64_t c1 = !in_ok ? c0 : (c0 + slice < cols) ? c0 + slice : cols;
  const int64_t piece = (int64_t)T * E;
  const bool resident = (c1 - c0) <= piece;

  float v[E];
  ML st{-INFINITY, 0.f};
  if (resident) {
    load_piece<E, VEC, true>(xr, c0, c1, v);
    st = thread_stats<E>(v);
  } else {
    for (int64_t b = c0; b < c1; b += piece) {
      load_piece<E, VEC, false>(xr, b, c1, v);
      st = ml_merge(st, thread_stats<E>(v));
    }
  }

  // warps -> CTA
  st = warp_merge(st);
  if (lane == 0) warp_ml[warp] = st;
  __syncthreads();
  if (warp == 0) {
    ML w = (lane < T / 32) ? warp_ml[lane] : ML{-INFINITY, 0.f};
    w = warp_merge(w);
    if (lane == 0) cta_ml = w;
  }
  __syncthreads();

  // CTAs of the cluster -> row (every CTA merges the slices in the same order, so all of them hold
  // bit-identical statistics): thread 0 reads the peers' pairs in rank order, or (PAR) lane r of
  // warp 0 reads peer r's pair, so that all the remote loads are in flight at once, and a shuffle
  // tree merges them (256 x 262,144: 4.89 -> 5.11 TB/s; in the 4-CTA instance the parallel form
  // measured 0.4 % slower).
  if (cluster > 1) {
    cluster_barrier();
    const uint32_t a = smem_addr(&cta_ml);
    if constexpr (PAR) {
      if (warp == 0) {
        ML pr{-INFINITY, 0.f};
        if (lane < cluster) pr = ML{ld_dsmem_f32(a, (uint32_t)lane), ld_dsmem_f32(a + 4, (uint32_t)lane)};
        pr = warp_merge(pr);
        if (lane == 0) row_ml = pr;
      }
    } else if (t == 0) {
      ML tot{-INFINITY, 0.f};
      for (int r = 0; r < cluster; ++r) tot = ml_merge(tot, ML{ld_dsmem_f32(a, r), ld_dsmem_f32(a + 4, r)});
      row_ml = tot;
    }
  } else if (t == 0) {
    row_ml = cta_ml;
  }
  __syncthreads();
  if (cluster > 1) cluster_arrive_relaxed();  // the remote reads are complete
  const ML rs = row_ml;

  if (lse != nullptr && rank == 0 && t == 0) lse[row] = (rs.l > 0.f) ? rs.m + logf(rs.l) : -INFINITY;

  if (y != nullptr) {
    const float inv_l = (rs.l > 0.f) ? 1.f / rs.l : 0.f;
    const float ref = (rs.m == -INFINITY) ? 0.f : rs.m;
    float* yr = y + row * ld_y;
    if (resident) {
      store_piece<E, VEC>(yr, c0, c1, v, ref, inv_l);
    } else {
      // the statistics pass ended on the slice's last piece, still in registers: it goes out
      // first, without a second read; the earlier pieces are read again (from L2)
      const int64_t last = c0 + (c1 - c0 - 1) / piece * piece;
      store_piece<E, VEC>(yr, last, c1, v, ref, inv_l);
      for (int64_t b = c0; b < last; b += piece) {
        load_piece<E, VEC, false>(xr, b, c1, v);
        store_piece<E, VEC>(yr, b, c1, v, ref, inv_l);
      }
    }
  }
  // keep this CTA's shared memory alive until every peer has read it
  if (cluster > 1) cluster_wait();
}

template <int E, bool VEC, bool PAR = false>
cudaError_t launch_cfg(const float* x, int64_t rows, int64_t cols, int64_t ld_x, float* y, int64_t ld_y,
                       float* lse, int threads, int cluster, int64_t slice, const DevStatus& st, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(rows * cluster), 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (cluster > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, softmax_rows_kernel<E, VEC, PAR>, x, rows, cols, ld_x, y, ld_y, lse, cluster, slice,
                            st);
}

constexpr int kMaxDevices = 64;

// Largest cluster the 32-element instance may use on the current device: 16 when the device
// schedules a non-portable cluster of that size for it, else the portable 8.
template <bool VEC>
int wide_cluster_limit(cudaStream_t s) {
  static int limit[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 8;
  if (limit[dev] == 0) {
    int lim = 8;
    if (cudaFuncSetAttribute(softmax_rows_kernel<32, VEC, true>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
        cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(16, 1, 1);
      cfg.blockDim = dim3(kMaxThreads, 1, 1);
      cfg.stream = s;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 16;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, softmax_rows_kernel<32, VEC, true>, &cfg) == cudaSuccess && n > 0) lim = 16;
    }
    (void)cudaGetLastError();  // a refused query leaves no error behind
    limit[dev] = lim;
  }
  return limit[dev];
}

template <bool VEC>
cudaError_t launch_vec(const float* x, int64_t rows, int64_t cols, int64_t ld_x, float* y, int64_t ld_y,
                       float* lse, const DevStatus& st, cudaStream_t s) {
  // Register capacity of one CTA: 256 threads x 32 fp32.  Up to 8 CTAs (a portable cluster) hold a
  // row on chip; wider rows take slices of two pieces, up to 16 CTAs a row (see the file comment).
  constexpr int64_t kCtaCap = (int64_t)kMaxThreads * 32;
  if (cols <= 1024) {
    const int threads = (int)(((cols + 3) / 4 + 31) / 32 * 32);
    return launch_cfg<4, VEC>(x, rows, cols, ld_x, y, ld_y, lse, threads, 1, (cols + 3) / 4 * 4, st, s);
  }
  if (cols <= 2048) return launch_cfg<8, VEC>(x, rows, cols, ld_x, y, ld_y, lse, kMaxThreads, 1, cols, st, s);
  if (cols <= 4096) return launch_cfg<16, VEC>(x, rows, cols, ld_x, y, ld_y, lse, kMaxThreads, 1, cols, st, s);
  int cluster = (int)((cols + kCtaCap - 1) / kCtaCap);
  if (cluster > 8) {
    cluster = (int)((cols + 2 * kCtaCap - 1) / (2 * kCtaCap));
    if (cluster > 8) {
      const int lim = wide_cluster_limit<VEC>(s);
      if (cluster > lim) cluster = lim;
    }
  }
  const int64_t slice = ((cols + cluster - 1) / cluster + 3) / 4 * 4;
  if (cluster > 4) return launch_cfg<32, VEC, true>(x, rows, cols, ld_x, y, ld_y, lse, kMaxThreads, cluster, slice, st, s);
  return launch_cfg<32, VEC>(x, rows, cols, ld_x, y, ld_y, lse, kMaxThreads, cluster, slice, st, s);
}

}  // namespace

cudaError_t launch_softmax_rows(const float* x, int64_t rows, int64_t cols, int64_t ld_x, float* y,
                                int64_t ld_y, float* lse, const DevStatus& st, cudaStream_t s) {
  const bool vec = (reinterpret_cast<uintptr_t>(x) % 16 == 0) && (ld_x % 4 == 0) &&
                   (y == nullptr || ((reinterpret_cast<uintptr_t>(y) % 16 == 0) && (ld_y % 4 == 0)));
  return vec ? launch_vec<true>(x, rows, cols, ld_x, y, ld_y, lse, st, s)
             : launch_vec<false>(x, rows, cols, ld_x, y, ld_y, lse, st, s);
}

}  // namespace oa
