// attn_splitkv.cu -- split-KV (decode style) attention partials.
//
// Interview lesson Step 5: with one query per row, splitting over queries
// leaves the GPU idle, so the keys are split instead.  One CTA per
// (row, chunk of keys) runs the online recurrence over its chunk and writes
// the chunk's normalised output o_c and lse_c; lse_merge.cu then merges
// the partials (Step 1's merge, log-sum-exp form).
//
// The chunk is streamed with 128-bit read-only loads: a key row of d
// elements is spread over d*size/16 lanes ("lanes per key"), so one warp
// reads several consecutive key rows -- a contiguous, coalesced span -- per
// load.  Each key group keeps its own running (m, l, o) with
// alpha = exp(m_old - m_new) rescaling (roadmap page s.5), updated once per
// U keys; the groups' states are merged with warp shuffles and then across
// warps through shared memory.  Scores are kept in log2 units (the scale is
// folded with log2 e into q), so each exponential is one ex2.
// Keys at or beyond kv_len[b] are never read; a chunk with no visible key
// writes o_c = 0, lse_c = -inf.  With grouped key/value heads (a KV cache
// with H / H_kv query heads per key/value head) one CTA serves the whole
// group: every K/V row is read once and scored against each of its queries.
#include "oa_internal.h"

namespace oa {
namespace {

constexpr int kWarps = 4;
constexpr int kU = 4;  // keys per group per step

__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

template <typename T>
struct Lanes;
template <>
struct Lanes<__nv_bfloat16> {
  static constexpr int kPerLane = 8;
  __device__ static void unpack(const uint4& u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};
template <>
struct Lanes<float> {
  static constexpr int kPerLane = 4;
  __device__ static void unpack(const uint4& u, float (&f)[4]) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
};

template <int EPL>
struct State {
  float m, l;
  float o[EPL];
};

template <int EPL>
__device__ __forceinline__ void merge_state(State<EPL>& a, float m2, float l2, const float (&o2)[EPL]) {
  const float m = fmaxf(a.m, m2);
  const float ref = (m == -INFINITY) ? 0.f : m;
  const float a1 = ex2(a.m - ref), a2 = ex2(m2 - ref);
  a.l = a.l * a1 + l2 * a2;
#pragma unroll
  for (int e = 0; e < EPL; ++e) a.o[e] = a.o[e] * a1 + o2[e] * a2;
  a.m = m;
}

// grid.x = R * S  (row-major over (row, chunk)); 128 threads.
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) splitkv_partial_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, float* __restrict__ part_o,
    float* __restrict__ part_lse, int H, int Nq, int Nk, int chunk, int S, float scale_log2,
    const int32_t* __restrict__ kv_len, int64_t R, int group) {
  constexpr int EPL = Lanes<T>::kPerLane;  // elements per lane (16 bytes)
  constexpr int LPK = D / EPL;             // lanes per key row
  constexpr int G = 32 / LPK;              // key rows per warp load
  constexpr int NG = kWarps * G;           // key groups in the CTA
  static_assert(LPK >= 1 && LPK <= 32 && (32 % LPK) == 0, "unsupported head dim");

  __shared__ float sm_m[kWarps], sm_l[kWarps];
  __shared__ float sm_o[kWarps][D];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t row = blockIdx.x / S;
  const int c = (int)(blockIdx.x % S);
  const int64_t bh = row / Nq;
  const int b = (int)(bh / H);
  int kvl = Nk;
  if (kv_len != nullptr) kvl = min(max(kv_len[b], 0), Nk);
  const int j0 = c * chunk;
  const int j1 = min(kvl, j0 + chunk);
  float* out_o = part_o + ((int64_t)c * R + row) * D;

  if (j0 >= j1) {  // empty chunk: zero weight in the merge
    for (int e = threadIdx.x; e < D; e += kWarps * 32) out_o[e] = 0.f;
    if (threadIdx.x == 0) part_lse[(int64_t)c * R + row] = -INFINITY;
    return;
  }

  const int sub = lane % LPK;            // which 16-byte piece of the row
  const int grp = warp * G + lane / LPK; // key group

  float qv[EPL];
  Lanes<T>::unpack(*reinterpret_cast<const uint4*>(q + row * D + sub * EPL), qv);
#pragma unroll
  for (int e = 0; e < EPL; ++e) qv[e] *= scale_log2;

  State<EPL> st;
  st.m = -INFINITY;
  st.l = 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) st.o[e] = 0.f;

  // query head h reads key/value head h / group
  const int64_t kvbh = (int64_t)b * (H / group) + (int)(bh % H) / group;
  const T* kb = k + (kvbh * Nk) * (int64_t)D + sub * EPL;
  const T* vb = v + (kvbh * Nk) * (int64_t)D + sub * EPL;

  for (int base = j0; base < j1; base += NG * kU) {
    uint4 kr[kU], vr[kU];
    bool ok[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int j = base + u * NG + grp;
      ok[u] = j < j1;
      if (ok[u]) {
        kr[u] = ld_stream(kb + (int64_t)j * D);
        vr[u] = ld_stream(vb + (int64_t)j * D);
      }
    }
    float s[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      float kf[EPL];
      Lanes<T>::unpack(ok[u] ? kr[u] : make_uint4(0, 0, 0, 0), kf);
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) dot = fmaf(qv[e], kf[e], dot);
#pragma unroll
      for (int off = LPK / 2; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      s[u] = ok[u] ? dot : -INFINITY;
    }
    float mt = s[0];
#pragma unroll
    for (int u = 1; u < kU; ++u) mt = fmaxf(mt, s[u]);
    const float m_new = fmaxf(st.m, mt);
    const float ref = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = ex2(st.m - ref);
    st.l *= alpha;
#pragma unroll
    for (int e = 0; e < EPL; ++e) st.o[e] *= alpha;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const float p = ex2(s[u] - ref);
      st.l += p;
      float vf[EPL];
      Lanes<T>::unpack(ok[u] ? vr[u] : make_uint4(0, 0, 0, 0), vf);
#pragma unroll
      for (int e = 0; e < EPL; ++e) st.o[e] = fmaf(p, vf[e], st.o[e]);
    }
    st.m = m_new;
  }

  // merge the G groups of this warp (lanes with the same `sub`)
#pragma unroll
  for (int off = LPK; off < 32; off <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, st.m, off);
    const float l2 = __shfl_xor_sync(0xffffffffu, st.l, off);
    float o2[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) o2[e] = __shfl_xor_sync(0xffffffffu, st.o[e], off);
    merge_state(st, m2, l2, o2);
  }
  if (lane < LPK) {
#pragma unroll
    for (int e = 0; e < EPL; ++e) sm_o[warp][sub * EPL + e] = st.o[e];
    if (lane == 0) {
      sm_m[warp] = st.m;
      sm_l[warp] = st.l;
    }
  }
  __syncthreads();
  // across warps, in warp order
  if (warp == 0) {
    float m = sm_m[0];
    for (int w = 1; w < kWarps; ++w) m = fmaxf(m, sm_m[w]);
    const float ref = (m == -INFINITY) ? 0.f : m;
    float l = 0.f, sc[kWarps];
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      sc[w] = ex2(sm_m[w] - ref);
      l += sm_l[w] * sc[w];
    }
    const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
    for (int e = lane; e < D; e += 32) {
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) acc += sm_o[w][e] * sc[w];
      out_o[e] = acc * inv_l;
    }
    if (lane == 0) part_lse[(int64_t)c * R + row] = (l > 0.f) ? (m + log2f(l)) * kLn2 : -INFINITY;
  }
}

// Grouped key/value heads: grid.x = (R / NQ) * S; one (b, key/value head, i) per CTA, whose NQ
// (= group) query heads share every K/V load, each with its own running (m, l, o).  The same
// recurrence and merges as splitkv_partial_kernel, NQ-wide.
template <typename T, int D, int NQ>
__global__ void __launch_bounds__(kWarps * 32) splitkv_group_kernel(
    const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v, float* __restrict__ part_o,
    float* __restrict__ part_lse, int H, int Nq, int Nk, int chunk, int S, float scale_log2,
    const int32_t* __restrict__ kv_len, int64_t R, int group) {
  constexpr int EPL = Lanes<T>::kPerLane;  // elements per lane (16 bytes)
  constexpr int LPK = D / EPL;             // lanes per key row
  constexpr int G = 32 / LPK;              // key rows per warp load
  constexpr int NG = kWarps * G;           // key groups in the CTA
  constexpr int KU = NQ >= 8 ? 2 : kU;  // keys per group per step (registers)
  static_assert(LPK >= 1 && LPK <= 32 && (32 % LPK) == 0, "unsupported head dim");

  __shared__ float sm_m[NQ][kWarps], sm_l[NQ][kWarps];
  __shared__ float sm_o[NQ][kWarps][D];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t crow = blockIdx.x / S;
  const int c = (int)(blockIdx.x % S);
  int64_t rows[NQ];
  int b;
  int64_t kvbh;  // key/value plane b H_kv + head
  static_assert(NQ > 1, "one query head per CTA is splitkv_partial_kernel");
  {
    const int Hkv = H / group;
    const int qi = (int)(crow % Nq);
    kvbh = crow / Nq;
    b = (int)(kvbh / Hkv);
    const int hkv = (int)(kvbh % Hkv);
#pragma unroll
    for (int t = 0; t < NQ; ++t) rows[t] = ((int64_t)b * H + hkv * NQ + t) * Nq + qi;
  }
  int kvl = Nk;
  if (kv_len != nullptr) kvl = min(max(kv_len[b], 0), Nk);
  const int j0 = c * chunk;
  const int j1 = min(kvl, j0 + chunk);

  if (j0 >= j1) {  // empty chunk: zero weight in the merge
#pragma unroll
    for (int t = 0; t < NQ; ++t) {
      float* out_o = part_o + ((int64_t)c * R + rows[t]) * D;
      for (int e = threadIdx.x; e < D; e += kWarps * 32) out_o[e] = 0.f;
      if (threadIdx.x == 0) part_lse[(int64_t)c * R + rows[t]] = -INFINITY;
    }
    return;
  }

  const int sub = lane % LPK;            // which 16-byte piece of the row
  const int grp = warp * G + lane / LPK; // key group

  float qv[NQ][EPL];
  State<EPL> st[NQ];
#pragma unroll
  for (int t = 0; t < NQ; ++t) {
    Lanes<T>::unpack(*reinterpret_cast<const uint4*>(q + rows[t] * D + sub * EPL), qv[t]);
#pragma unroll
    for (int e = 0; e < EPL; ++e) qv[t][e] *= scale_log2;
    st[t].m = -INFINITY;
    st[t].l = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) st[t].o[e] = 0.f;
  }

  const T* kb = k + (kvbh * Nk) * (int64_t)D + sub * EPL;
  const T* vb = v + (kvbh * Nk) * (int64_t)D + sub * EPL;

  for (int base = j0; base < j1; base += NG * KU) {
    uint4 kr[KU], vr[KU];
    bool ok[KU];
#pragma unroll
    for (int u = 0; u < KU; ++u) {
      const int j = base + u * NG + grp;
      ok[u] = j < j1;
      if (ok[u]) {
        kr[u] = ld_stream(kb + (int64_t)j * D);
        vr[u] = ld_stream(vb + (int64_t)j * D);
      }
    }
    float s[KU][NQ];
#pragma unroll
    for (int u = 0; u < KU; ++u) {
      float kf[EPL];
      Lanes<T>::unpack(ok[u] ? kr[u] : make_uint4(0, 0, 0, 0), kf);
#pragma unroll
      for (int t = 0; t < NQ; ++t) {
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) dot = fmaf(qv[t][e], kf[e], dot);
#pragma unroll
        for (int off = LPK / 2; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        s[u][t] = ok[u] ? dot : -INFINITY;
      }
    }
    float vf[KU][EPL];  // each V row unpacked once for all the group's query heads
#pragma unroll
    for (int u = 0; u < KU; ++u) Lanes<T>::unpack(ok[u] ? vr[u] : make_uint4(0, 0, 0, 0), vf[u]);
#pragma unroll
    for (int t = 0; t < NQ; ++t) {
      float mt = s[0][t];
#pragma unroll
      for (int u = 1; u < KU; ++u) mt = fmaxf(mt, s[u][t]);
      const float m_new = fmaxf(st[t].m, mt);
      const float ref = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2(st[t].m - ref);
      st[t].l *= alpha;
#pragma unroll
      for (int e = 0; e < EPL; ++e) st[t].o[e] *= alpha;
#pragma unroll
      for (int u = 0; u < KU; ++u) {
        const float p = ex2(s[u][t] - ref);
        st[t].l += p;
#pragma unroll
        for (int e = 0; e < EPL; ++e) st[t].o[e] = fmaf(p, vf[u][e], st[t].o[e]);
      }
      st[t].m = m_new;
    }
  }

#pragma unroll
  for (int t = 0; t < NQ; ++t) {
    // merge the G groups of this warp (lanes with the same `sub`)
#pragma unroll
    for (int off = LPK; off < 32; off <<= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, st[t].m, off);
      const float l2 = __shfl_xor_sync(0xffffffffu, st[t].l, off);
      float o2[EPL];
#pragma unroll
      for (int e = 0; e < EPL; ++e) o2[e] = __shfl_xor_sync(0xffffffffu, st[t].o[e], off);
      merge_state(st[t], m2, l2, o2);
    }
    if (lane < LPK) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) sm_o[t][warp][sub * EPL + e] = st[t].o[e];
      if (lane == 0) {
        sm_m[t][warp] = st[t].m;
        sm_l[t][warp] = st[t].l;
      }
    }
  }
  __syncthreads();
  // across warps, in warp order; warp t % kWarps finishes query head t
#pragma unroll
  for (int t = 0; t < NQ; ++t) {
    if (warp != t % kWarps) continue;
    float m = sm_m[t][0];
    for (int w = 1; w < kWarps; ++w) m = fmaxf(m, sm_m[t][w]);
    const float ref = (m == -INFINITY) ? 0.f : m;
    float l = 0.f, sc[kWarps];
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      sc[w] = ex2(sm_m[t][w] - ref);
      l += sm_l[t][w] * sc[w];
    }
    const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
    float* out_o = part_o + ((int64_t)c * R + rows[t]) * D;
    for (int e = lane; e < D; e += 32) {
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) acc += sm_o[t][w][e] * sc[w];
      out_o[e] = acc * inv_l;
    }
    if (lane == 0) part_lse[(int64_t)c * R + rows[t]] = (l > 0.f) ? (m + log2f(l)) * kLn2 : -INFINITY;
  }
}

template <typename T, int D, int NQ>
cudaError_t launch_group(const void* q, const void* k, const void* v, int64_t R, int H, int Nq, int Nk, int S,
                         float scale, const int32_t* kv_len, float* part_o, float* part_lse, int group,
                         cudaStream_t s) {
  const int chunk = (Nk + S - 1) / S;
  splitkv_group_kernel<T, D, NQ><<<(unsigned)(R / NQ * S), kWarps * 32, 0, s>>>(
      static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), part_o, part_lse, H, Nq, Nk,
      chunk, S, scale * kLog2e, kv_len, R, group);
  return cudaGetLastError();
}

// Query heads of a group share K/V loads for the usual decode head sizes; other sizes (and
// H_kv == H) run one query head per CTA.
template <typename T, int D>
cudaError_t launch_t(const void* q, const void* k, const void* v, int64_t R, int H, int Nq, int Nk, int S,
                     float scale, const int32_t* kv_len, float* part_o, float* part_lse, int group, cudaStream_t s) {
  if constexpr (D >= 64 && (sizeof(T) == 2 || D <= 128)) {
    switch (group) {
      case 2: return launch_group<T, D, 2>(q, k, v, R, H, Nq, Nk, S, scale, kv_len, part_o, part_lse, group, s);
      case 4: return launch_group<T, D, 4>(q, k, v, R, H, Nq, Nk, S, scale, kv_len, part_o, part_lse, group, s);
      case 8: return launch_group<T, D, 8>(q, k, v, R, H, Nq, Nk, S, scale, kv_len, part_o, part_lse, group, s);
      default: break;
    }
  }
  const int chunk = (Nk + S - 1) / S;
  splitkv_partial_kernel<T, D><<<(unsigned)(R * S), kWarps * 32, 0, s>>>(
      static_cast<const T*>(q), static_cast<const T*>(k), static_cast<const T*>(v), part_o, part_lse, H, Nq, Nk,
      chunk, S, scale * kLog2e, kv_len, R, group);
  return cudaGetLastError();
}

}  // namespace

bool splitkv_supported(bool bf16, int d) {
  if (bf16) return d == 8 || d == 16 || d == 32 || d == 64 || d == 128 || d == 256;
  return d == 4 || d == 8 || d == 16 || d == 32 || d == 64 || d == 128;
}

cudaError_t launch_splitkv_partial(const void* q, const void* k, const void* v, bool bf16, int B, int H, int Hkv,
                                   int Nq, int Nk, int d, float scale, const int32_t* kv_len, int S, float* part_o,
                                   float* part_lse, cudaStream_t s) {
  const int64_t R = (int64_t)B * H * Nq;
  const int group = H / Hkv;
  using bf = __nv_bfloat16;
  if (bf16) {
    switch (d) {
      case 8: return launch_t<bf, 8>(q, k, v, R, H, Nq, Nk, S, scale, kv_len, part_o, part_lse, group, s);
      case 16: return launch_t<bf, 16>(q, k, v, R, H, Nq, Nk, S, scale, kv_len, part_o, part_lse, group, s);
      case 32: return launch_t<bf, 32>(q, k, v, R, H, Nq, Nk, S, scale, kv_len, part_o, part_lse, group, s);
      case 64: return launch_t<bf, 64>(q, k, v, R, H, Nq, Nk, S, scale, kv_len, part_o, part_lse, group, s);
      case 128: return launch_t<bf, 128>(q, k, v, R, H, Nq, Nk, S, scale, kv_len, part_o, part_lse, group, s);
      case 256: return launch_t<bf, 256>(q, k, v, R, H, Nq, Nk, S, scale, kv_len, part_o, part_lse, group, s);
    }
  } else {
    switch (d) {
      case 4: return launch_t<float, 4>(q, k, v, R, H, Nq, Nk, S, scale, kv_len, part_o, part_lse, group, s);
      case 8: return launch_t<float, 8>(q, k, v, R, H, Nq, Nk, S, scale, kv_len, part_o, part_lse, group, s);
      case 16: return launch_t<float, 16>(q, k, v, R, H, Nq, Nk, S, scale, kv_len, part_o, part_lse, group, s);
      case 32: return launch_t<float, 32>(q, k, v, R, H, Nq, Nk, S, scale, kv_len, part_o, part_lse, group, s);
      case 64: return launch_t<float, 64>(q, k, v, R, H, Nq, Nk, S, scale, kv_len, part_o, part_lse, group, s);
      case 128: return launch_t<float, 128>(q, k, v, R, H, Nq, Nk, S, scale, kv_len, part_o, part_lse, group, s);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace oa
