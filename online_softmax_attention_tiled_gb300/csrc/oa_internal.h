// oa_internal.h -- launchers implemented by each kernel translation unit
// and called by the C ABI layer (oa_api.cu).  Arguments have already been
// validated there; launchers only pick a configuration and launch.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "oa_common.cuh"

namespace oa {

cudaError_t launch_softmax_rows(const float* x, int64_t rows, int64_t cols, int64_t ld_x, float* y,
                                int64_t ld_y, float* lse, const DevStatus& st, cudaStream_t s);

cudaError_t launch_lse_merge(const float* part_o, const float* part_lse, int S, int64_t R, int d, void* o,
                             bool o_bf16, float* lse, cudaStream_t s);

cudaError_t launch_attn_f32(const float* q, const float* k, const float* v, float* o, float* lse, int B,
                            int H, int Hkv, int Nq, int Nk, int d, int causal, float scale, const int32_t* kv_len,
                            int Br, int Bc, cudaStream_t s);

// True if (bf16, d) / (fp32, d) has a split-KV partial kernel.
bool splitkv_supported(bool bf16, int d);
// K/V have Hkv heads; query head h reads head h / (H / Hkv).
cudaError_t launch_splitkv_partial(const void* q, const void* k, const void* v, bool bf16, int B, int H, int Hkv,
                                   int Nq, int Nk, int d, float scale, const int32_t* kv_len,
                                   int num_splits, float* part_o, float* part_lse, cudaStream_t s);

// bf16 rows of D elements viewed as a 3-D tensor for TMA (D innermost, then `rows` rows
// `row_bytes` apart, then `planes` planes `plane_bytes` apart); box 64 x box_rows x 1 with the
// 128-byte swizzle; reads past the end return zero.  False if the encoder is unavailable or
// rejects the layout.
bool make_tile_map(CUtensorMap* map, const void* base, int D, int rows, int64_t row_bytes, int planes,
                   int64_t plane_bytes, int box_rows = 128);
// fp32 [planes][rows][cols], box {32, box_rows, 1}, 128-byte swizzle (TMA reduce-add targets).
bool make_f32_tile_map(CUtensorMap* map, const void* base, int cols, int rows, int64_t row_bytes, int planes,
                       int64_t plane_bytes, int box_rows);

// Tensor-core attention (tcgen05 + TMA), bf16, d in {64, 128}.
//   dense  (cu_q == NULL): q/o [B, H, Nq, d], k/v [B, Hkv, Nk, d], kv_len[B] or NULL.
//   packed (cu_q != NULL): B sequences; q/o [Tq, H, d], k/v [Tk, Hkv, d], lse [Tq, H];
//          sequence s has query tokens [cu_q[s], cu_q[s+1]) and key tokens [cu_k[s], cu_k[s+1]);
//          Nq / Nk are the longest query / key sequence.
// Query head h reads key/value head h / (H / Hkv).
struct TcArgs {
  const void *q, *k, *v;
  void* o;
  float* lse;
  int B, H, Hkv, Nq, Nk, d, causal;
  float scale;
  const int32_t* kv_len;
  const int32_t *cu_q, *cu_k;
  int Tq, Tk;
  // > 0: the rows of a plane are the queries of several query heads, qmod each (grouped decode); a
  // row's causal position is its index modulo qmod, and Nk - qmod is the causal key offset
  int qmod;
  // Dense: this launch computes planes [order_sh0, order_sh0 + B H) of a call of order_bh planes
  // cut into pieces (0: the launch is the whole call); the order of each item's key tiles is that
  // of the whole call, so the pieces give its results bit for bit
  int order_bh, order_sh0;
};
// `why` gets a static message when the host-side set-up (tensor maps) fails.
cudaError_t launch_attn_tc(const TcArgs& a, const DevStatus& st, cudaStream_t s, const char** why);

// Attention backward (tcgen05 + TMA), bf16, d in {64, 128}, dense [B, H, N, d] layouts:
// dq/do/q [B, H, Nq, d], dk/dv/k/v [B, H, Nk, d], lse [B, H, Nq] from the forward.
struct BwdArgs {
  const void *q, *k, *v, *o, *dout;
  const float* lse;
  void *dq, *dk, *dv;
  int B, H, Hkv, Nq, Nk, d, causal;  // query head h reads key/value head h / (H / Hkv)
  float scale;
  // packed sequences (NULL for the dense layout): token-major [Nq, H, d] / [Nk, Hkv, d] tensors with
  // B = 1 and Nq, Nk the token counts; sequence s owns rows [cu[s], cu[s + 1])
  const int32_t *cu_q = nullptr, *cu_k = nullptr;
  int num_seqs = 0, max_seqlen_k = 0;
};
// fp32 values of workspace the backward needs: the dQ accumulator [B H Nq, d] and D [B H Nq].
size_t attn_bwd_workspace_floats(int B, int H, int Nq, int d);
// Three launches on `s` (pre-pass, main kernel, dQ conversion).  `why` as for launch_attn_tc.
cudaError_t launch_attn_bwd(const BwdArgs& a, float* workspace, const DevStatus& st, cudaStream_t s,
                            const char** why);

cudaError_t launch_selftest_wait(const DevStatus& st, cudaStream_t s);
cudaError_t launch_selftest_check(const DevStatus& st, int* out, cudaStream_t s);

}  // namespace oa
