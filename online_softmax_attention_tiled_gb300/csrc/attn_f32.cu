// attn_f32.cu -- fp32 attention forward on the CUDA cores with runtime tile
// sizes (Br query rows per CTA, Bc keys per step).
//
// The tile recurrence of the roadmap page (s.4, s.5) in the Q-outer order
// (interview lesson Step 3): each CTA holds one block of Br query rows and
// their running state (m, l, o) and streams the key/value blocks past it:
//   m_new = max(m_old, max_c s_c),  alpha = exp(m_old - m_new),
//   p_c = exp(s_c - m_new),  l = alpha l + sum p,  o = alpha o + sum p_c v_c,
// with one normalisation o / l at the end and LSE = m + ln l.  Masked
// scores are -inf; a row that has seen nothing keeps m = -inf and uses 0 as
// its reference, so alpha and p are exactly 0 and no NaN forms.
// Causal: the Nq queries are the last Nq positions of the Nk keys' sequence,
// so query i sees keys j <= i + (Nk - Nq) (j <= i when Nq == Nk).  Causal
// CTAs stop at their last visible key block (blocks past the diagonal are
// skipped; the blocks it crosses are masked element-wise).
#include "oa_internal.h"

namespace oa {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) attn_f32_kernel(const float* __restrict__ q,
                                                            const float* __restrict__ k,
                                                            const float* __restrict__ v, float* __restrict__ o,
                                                            float* __restrict__ lse, int H, int Nq, int Nk, int d,
                                                            int causal, float scale,
                                                            const int32_t* __restrict__ kv_len, int Br, int Bc,
                                                            int n_qblocks, int group) {
  extern __shared__ float sm[];
  float* Qs = sm;                 // [Br][d]
  float* Os = Qs + Br * d;        // [Br][d]
  float* Ks = Os + Br * d;        // [Bc][d]
  float* Vs = Ks + Bc * d;        // [Bc][d]
  float* Ss = Vs + Bc * d;        // [Br][Bc]
  float* ms = Ss + Br * Bc;       // [Br]
  float* ls = ms + Br;            // [Br]
  float* as = ls + Br;            // [Br]

  const int t = threadIdx.x, lane = t & 31, warp = t >> 5, nwarps = kThreads / 32;
  const int64_t bh = blockIdx.x / n_qblocks;
  const int q0 = (int)(blockIdx.x % n_qblocks) * Br;
  const int b = (int)(bh / H);
  int kvl = Nk;
  if (kv_len != nullptr) kvl = min(max(kv_len[b], 0), Nk);
  const int br = min(Br, Nq - q0);
  const int off = Nk - Nq;  // causal: query i sees keys j <= i + off
  const int kv_end = causal ? min(kvl, max(0, q0 + br + off)) : kvl;

  const float* qb = q + (bh * Nq + q0) * d;
  // query head h reads key/value head h / group
  const int64_t kvbh = (int64_t)b * (H / group) + (int)(bh % H) / group;
  const float* kb = k + kvbh * (int64_t)Nk * d;
  const float* vb = v + kvbh * (int64_t)Nk * d;

  for (int i = t; i < br * d; i += kThreads) {
    Qs[i] = qb[i];
    Os[i] = 0.f;
  }
  for (int r = t; r < br; r += kThreads) {
    ms[r] = -INFINITY;
    ls[r] = 0.f;
  }

  for (int j0 = 0; j0 < kv_end; j0 += Bc) {
    const int bc = min(Bc, kv_end - j0);
    __syncthreads();  // previous step's users of Ks/Vs/Ss are done
    for (int i = t; i < bc * d; i += kThreads) {
      Ks[i] = kb[(int64_t)j0 * d + i];
      Vs[i] = vb[(int64_t)j0 * d + i];
    }
    __syncthreads();
    // scores of this (Q block, KV block) pair
    for (int i = t; i < br * bc; i += kThreads) {
      const int r = i / bc, c = i % bc;
      const int col = j0 + c, row = q0 + r;
      float s = -INFINITY;
      if (col < kvl && (!causal || col <= row + off)) {
        float acc = 0.f;
        for (int e = 0; e < d; ++e) acc = fmaf(Qs[r * d + e], Ks[c * d + e], acc);
        s = acc * scale;
      }
      Ss[r * Bc + c] = s;
    }
    __syncthreads();
    // per-row state update, one warp per row
    for (int r = warp; r < br; r += nwarps) {
      float mt = -INFINITY;
      for (int c = lane; c < bc; c += 32) mt = fmaxf(mt, Ss[r * Bc + c]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
      const float m_old = ms[r];
      const float m_new = fmaxf(m_old, mt);
      const float ref = (m_new == -INFINITY) ? 0.f : m_new;
      float psum = 0.f;
      for (int c = lane; c < bc; c += 32) {
        const float p = expf(Ss[r * Bc + c] - ref);
        Ss[r * Bc + c] = p;
        psum += p;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
      if (lane == 0) {
        const float alpha = expf(m_old - ref);
        ls[r] = alpha * ls[r] + psum;
        ms[r] = m_new;
        as[r] = alpha;
      }
    }
    __syncthreads();
    // o = alpha o + P V
    for (int i = t; i < br * d; i += kThreads) {
      const int r = i / d, e = i % d;
      float acc = as[r] * Os[i];
      for (int c = 0; c < bc; ++c) acc = fmaf(Ss[r * Bc + c], Vs[c * d + e], acc);
      Os[i] = acc;
    }
  }
  __syncthreads();
  float* ob = o + (bh * Nq + q0) * d;
  for (int i = t; i < br * d; i += kThreads) {
    const int r = i / d;
    const float l = ls[r];
    ob[i] = (l > 0.f) ? Os[i] / l : 0.f;
  }
  if (lse != nullptr)
    for (int r = t; r < br; r += kThreads) {
      const float l = ls[r];
      lse[bh * Nq + q0 + r] = (l > 0.f) ? ms[r] + logf(l) : -INFINITY;
    }
}

size_t smem_bytes(int Br, int Bc, int d) {
  return sizeof(float) * ((size_t)2 * Br * d + (size_t)2 * Bc * d + (size_t)Br * Bc + 3 * (size_t)Br);
}

}  // namespace

cudaError_t launch_attn_f32(const float* q, const float* k, const float* v, float* o, float* lse, int B, int H,
                            int Hkv, int Nq, int Nk, int d, int causal, float scale, const int32_t* kv_len, int Br,
                            int Bc, cudaStream_t s) {
  if (Br <= 0 || Bc <= 0) {  // library default tiles
    Br = 16;
    Bc = 64;
  }
  const size_t smem = smem_bytes(Br, Bc, d);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(attn_f32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  const int n_qblocks = (Nq + Br - 1) / Br;
  const int64_t grid = (int64_t)B * H * n_qblocks;
  attn_f32_kernel<<<(unsigned)grid, kThreads, smem, s>>>(q, k, v, o, lse, H, Nq, Nk, d, causal, scale, kv_len,
                                                         Br, Bc, n_qblocks, H / Hkv);
  return cudaGetLastError();
}

}  // namespace oa
