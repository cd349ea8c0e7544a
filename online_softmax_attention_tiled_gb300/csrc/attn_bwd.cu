// attn_bwd.cu -- attention backward on the 5th-generation tensor cores (tcgen05, tensor
// memory, TMA), bf16 inputs, fp32 accumulation, d = 64 / 128.
//
// What it computes: the gradients of O = softmax(scale Q K^T) V for a given dO, with the
// attention weights recomputed from the scores and the forward's per-row LSE instead of
// being read back from a stored [N, N] matrix (page "Online softmax in attention -- why
// and how", "Where this is heading: FA2": on backward, recompute the scores from the cached
// softmax statistics).  With P = exp(scale S - LSE) (S = Q K^T, masked keys 0):
//   dV = P^T dO,   dP = dO V^T,   D = rowsum(dO o O),   dS = P o (dP - D),
//   dQ = scale dS K,   dK = scale dS^T Q.
//
// Three launches: a pre-pass (D per query row; the fp32 dQ accumulator zeroed), the main
// kernel, and a post-pass (dQ to bf16).  Main kernel, key-tile outer: one CTA per (b, h,
// 128 keys); K_j and V_j stay in shared memory while the query tiles i (causal: i >= j)
// stream through a 2-stage TMA ring with their dO tiles.  Per query tile:
//   S^T  = K_j Q_i^T,   dP^T = V_j dO_i^T           (SS MMAs into TMEM, lanes = keys)
//   P^T, dS^T  elementwise, one thread per key row  (P^T, dS^T as bf16 back into TMEM;
//                                                     dS^T also into shared memory)
//   dV_j += P^T dO_i,   dK_j += dS^T Q_i           (TS MMAs: A from TMEM, accumulate in TMEM)
//   dQ_i  = dS K_j                                   (SS MMA: A = the staged dS, read M-major)
// and the dQ_i tile is added into the fp32 accumulator in global memory (the tiles of
// other key blocks add into the same rows) by TMA reduce-adds of 32 x 32 blocks staged in
// shared memory.  dK_j, dV_j leave TMEM once, at the end.  The 128 (LSE log2 e, D) pairs
// of a query tile are loaded once per step into shared memory and read as broadcasts.
//
// GB300 mapping (320 threads, one CTA per SM):
//   warps 0-7  warp w reaches TMEM lanes 32 (w % 4) .. +31, so thread t owns key row t % 128
//              of the tile for the elementwise pass and the dK/dV epilogue, and query row
//              t % 128 of the dQ tile; warps 0-3 take queries (or columns) [0, 64), warps 4-7
//              [64, 128): two row warps per SM sub-partition
//   warp 8     TMA producer (K_j, V_j once; Q_i, dO_i per step)
//   warp 9     MMA issue (whole warp, one elected lane); owns the TMEM allocation
// TMEM (512 columns): S^T [0, 128) -> P^T bf16 (queries 0-63 in [0, 32), 64-127 in [64, 96),
// so neither half overwrites scores the other still reads) -> dQ_i fp32 [0, d); dP^T
// [128, 256) -> dS^T bf16 likewise at +128; dV [256, 256 + d); dK [256 + d, 256 + 2d).
//
// Every wait is bounded (oa_common.cuh); a wait that expires aborts the CTA, which falls
// through to its teardown with TMEM freed.
#include "oa_internal.h"

namespace oa {
namespace {

constexpr int BT = 128;                  // keys per CTA tile = query rows per step
constexpr int kBwdRowWarps = 8;
constexpr int kBwdThreads = 32 * (kBwdRowWarps + 2);
constexpr int kBwdProducer = kBwdRowWarps;
constexpr int kBwdMma = kBwdRowWarps + 1;
constexpr uint32_t kBwdTmemCols = 512;

template <int D>
struct BwdCfg {
  static constexpr int SLABS = D / 64;        // 128-byte swizzle atoms along d
  static constexpr int SLAB_BYTES = BT * 128;  // 128 rows x 128 bytes
  static constexpr int TILE_BYTES = SLABS * SLAB_BYTES;
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + TILE_BYTES;
  static constexpr int Q_OFF = V_OFF + TILE_BYTES;    // 2 stages
  static constexpr int DO_OFF = Q_OFF + 2 * TILE_BYTES;  // 2 stages
  // dS of one step, keys as rows and the 128 queries contiguous (two 64-query slabs): the
  // A operand of dQ = dS K read M-major
  static constexpr int ST_OFF = DO_OFF + 2 * TILE_BYTES;
  static constexpr int ST_BYTES = 2 * SLAB_BYTES;
  // (LSE log2 e, D) of the step's 128 query rows, float2 each (+inf / 0 past the end)
  static constexpr int LD_OFF = ST_OFF + ST_BYTES;
  static constexpr int BAR_OFF = LD_OFF + BT * 8;
  // kv_full, qdo_full[2], qdo_empty[2], s_full, dp_full, ds_ready, dq_full, dq_read, done, ld_ready
  static constexpr int NUM_BARS = 12;
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;  // + slack to align the base to 1024
  static constexpr uint32_t S_COL = 0, DP_COL = 128, DV_COL = 256, DK_COL = 256 + D;
  // S^T = K Q^T and dP^T = V dO^T: both operands K-major
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(BT, BT, false);
  // dV += P^T dO and dK += dS^T Q: A from TMEM, B (dO, Q with d contiguous) N-major
  static constexpr uint32_t IDESC_KV = idesc_bf16_f32(BT, D, true);
  // dQ = dS K: A (staged dS, queries contiguous) M-major, B (K, d contiguous) N-major
  static constexpr uint32_t IDESC_Q = idesc_bf16_f32(BT, D, true, true);
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

struct BwdParams {
  float* dq_acc;         // fp32 [B H Nq, d], zeroed by the pre-pass
  const float* lse;      // forward LSE [B H Nq]
  const float* dsum;     // D [B H Nq]
  __nv_bfloat16* dk;     // [B H Nk, d]
  __nv_bfloat16* dv;
  int Nq, Nk, causal, nkt, nqt, BH;
  float scale, scale_log2;
  DevStatus st;
};

enum BwdWait : unsigned { B_KV = 1, B_QDO, B_QDO_EMPTY, B_S, B_DP, B_DS, B_DQ, B_DQ_READ, B_DONE, B_LD };

// D[r] = sum_e dO[r, e] O[r, e] for every query row; dq_acc[r, :] = 0.  One warp per row.
__global__ void bwd_pre_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ dout,
                               float* __restrict__ dsum, float* __restrict__ dq_acc, int64_t rows, int d) {
  const int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const __nv_bfloat16* orow = o + r * d;
  const __nv_bfloat16* drow = dout + r * d;
  float acc = 0.f;
  for (int e = lane; e < d; e += 32) acc = fmaf(__bfloat162float(orow[e]), __bfloat162float(drow[e]), acc);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) dsum[r] = acc;
  float* qrow = dq_acc + r * d;
  for (int e = lane; e < d; e += 32) qrow[e] = 0.f;
}

// dq = bf16(dq_acc), four elements per thread (n is a multiple of 4).
__global__ void bwd_post_kernel(const float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dq, int64_t n) {
  const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (i >= n) return;
  const float4 a = *reinterpret_cast<const float4*>(dq_acc + i);
  uint2 w;
  w.x = pack_bf16x2(a.x, a.y);
  w.y = pack_bf16x2(a.z, a.w);
  *reinterpret_cast<uint2*>(dq + i) = w;
}

// P^T and dS^T for 32 queries q_first .. q_first + 31 of one key row: sr / dr the fp32 S^T and
// dP^T columns, ld the (LSE log2 e, D) pairs of those queries (two per float4).  MASK applies
// the key and causal tests as an exponent of -inf (no branch per element).
template <bool MASK>
__device__ __forceinline__ void bwd_p_ds(const uint32_t (&sr)[32], const uint32_t (&dr)[32], const float4* ld,
                                         float sl2, int key, int q_first, bool key_ok, bool causal,
                                         uint32_t (&pw)[16], uint32_t (&dw)[16]) {
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    const float4 l = ld[e / 2];  // a broadcast: every lane reads the same 16 bytes
    // P^T = exp(scale s - LSE) = exp2(s scale log2 e - LSE log2 e)
    float a0 = fmaf(__uint_as_float(sr[e]), sl2, -l.x);
    float a1 = fmaf(__uint_as_float(sr[e + 1]), sl2, -l.z);
    if (MASK) {
      const int q = q_first + e;
      a0 = (key_ok && (!causal || key <= q)) ? a0 : -INFINITY;
      a1 = (key_ok && (!causal || key <= q + 1)) ? a1 : -INFINITY;
    }
    const float p0 = ex2(a0), p1 = ex2(a1);
    pw[e / 2] = pack_bf16x2(p0, p1);
    dw[e / 2] = pack_bf16x2(p0 * (__uint_as_float(dr[e]) - l.y), p1 * (__uint_as_float(dr[e + 1]) - l.w));
  }
}

// grid.x = nkt * BH: blockIdx.x / BH is the key tile j (low j first: for causal those have
// the most query tiles), blockIdx.x % BH the (b, h) plane.
template <int D>
__global__ void __launch_bounds__(kBwdThreads)
    attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_addr(smem_raw);
  const uint32_t pad = (1024u - (raw_s & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_s + pad;

  const uint32_t bar0 = sbase + C::BAR_OFF;
  const uint32_t bar_kv = bar0;
  auto bar_qdo = [&](int s) { return bar0 + 8u * (1 + s); };        // Q_i, dO_i of stage s landed
  auto bar_qdo_empty = [&](int s) { return bar0 + 8u * (3 + s); };  // stage s read by its MMAs
  const uint32_t bar_s = bar0 + 8u * 5;        // S^T in TMEM
  const uint32_t bar_dp = bar0 + 8u * 6;       // dP^T in TMEM
  const uint32_t bar_ds = bar0 + 8u * 7;       // P^T, dS^T in TMEM and dS staged (4 warps)
  const uint32_t bar_dq = bar0 + 8u * 8;       // dQ_i in TMEM
  const uint32_t bar_dq_read = bar0 + 8u * 9;  // dQ_i read out of TMEM (4 warps)
  const uint32_t bar_done = bar0 + 8u * 10;    // every MMA of the CTA complete
  const uint32_t bar_ld = bar0 + 8u * 11;      // the step's (LSE, D) block written (4 warps)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = (int)(blockIdx.x / p.BH);
  const int bh = (int)(blockIdx.x % p.BH);
  const int k0 = j * BT;
  const int i_begin = p.causal ? j : 0;  // causal: query tile i sees key tile j iff i >= j
  const int n_it = max(p.nqt - i_begin, 0);

  if (threadIdx.x == 0) {
    mbar_init(bar_kv, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_qdo(s), 1);
      mbar_init(bar_qdo_empty(s), 1);
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_dp, 1);
    mbar_init(bar_ds, kBwdRowWarps);
    mbar_init(bar_dq, 1);
    mbar_init(bar_dq_read, kBwdRowWarps);
    mbar_init(bar_ld, kBwdRowWarps);
    mbar_init(bar_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kBwdMma) {
    tmem_alloc(smem_addr(tmem_slot), kBwdTmemCols);
    tmem_relinquish();
  }
  if (warp == kBwdProducer && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_dq);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  auto wait_all = [&](uint32_t bar, uint32_t parity, unsigned site) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, p.st, abort_flag, (K_ATTN_BWD << 8) | site));
  };

  if (warp == kBwdProducer) {
    // =================== TMA producer (whole warp, one elected lane issues) ===================
    bool ok = true;
    mbar_arrive_expect_tx_elect(bar_kv, 2 * C::TILE_BYTES);
    for (int c = 0; c < C::SLABS; ++c) {
      tma_load_3d_elect(sbase + C::K_OFF + c * C::SLAB_BYTES, &tm_k, bar_kv, c * 64, k0, bh);
      tma_load_3d_elect(sbase + C::V_OFF + c * C::SLAB_BYTES, &tm_v, bar_kv, c * 64, k0, bh);
    }
    int issued = 0;
    for (int it = 0; it < n_it; ++it) {
      const int s = it & 1, q0 = (i_begin + it) * BT;
      // stage s was last read by step it - 2
      if (it >= 2 && !(ok = wait_all(bar_qdo_empty(s), (uint32_t)((it >> 1) - 1) & 1u, B_QDO_EMPTY))) break;
      mbar_arrive_expect_tx_elect(bar_qdo(s), 2 * C::TILE_BYTES);
      for (int c = 0; c < C::SLABS; ++c) {
        tma_load_3d_elect(sbase + C::Q_OFF + s * C::TILE_BYTES + c * C::SLAB_BYTES, &tm_q, bar_qdo(s), c * 64, q0,
                          bh);
        tma_load_3d_elect(sbase + C::DO_OFF + s * C::TILE_BYTES + c * C::SLAB_BYTES, &tm_do, bar_qdo(s), c * 64,
                          q0, bh);
      }
      ++issued;
    }
    // drain: every load issued must have landed before the CTA can exit
    for (int it = max(0, issued - 2); it < issued; ++it)
      mbar_wait(bar_qdo(it & 1), (uint32_t)(it >> 1) & 1u, p.st, nullptr, (K_ATTN_BWD << 8) | B_DONE);
    mbar_wait(bar_kv, 0, p.st, nullptr, (K_ATTN_BWD << 8) | B_DONE);
  } else if (warp == kBwdMma) {
    // =================== MMA issue (whole warp, one elected lane) ===================
    const uint64_t k_kmaj = smem_desc_sw128(sbase + C::K_OFF, 16, 1024);   // A of S^T
    const uint64_t v_kmaj = smem_desc_sw128(sbase + C::V_OFF, 16, 1024);   // A of dP^T
    const uint64_t k_nmaj = smem_desc_sw128(sbase + C::K_OFF, C::SLAB_BYTES, 1024);  // B of dQ
    const uint64_t st_mmaj = smem_desc_sw128(sbase + C::ST_OFF, C::SLAB_BYTES, 1024);  // A of dQ
    auto kmaj_off = [](int kk) { return (uint64_t)(((kk / 4) * C::SLAB_BYTES + (kk % 4) * 32) >> 4); };
    auto rows16_off = [](int kk) { return (uint64_t)((kk * 16 * 128) >> 4); };  // 16 rows of 128 bytes
    auto pcol = [](int kk) { return (uint32_t)(kk * 8 + (kk >= 4 ? 32 : 0)); };  // P^T / dS^T column
    bool ok = wait_all(bar_kv, 0, B_KV);
    for (int it = 0; ok && it < n_it; ++it) {
      const int s = it & 1;
      const uint32_t ph = (uint32_t)it & 1u;
      const uint64_t q_kmaj = smem_desc_sw128(sbase + C::Q_OFF + s * C::TILE_BYTES, 16, 1024);
      const uint64_t do_kmaj = smem_desc_sw128(sbase + C::DO_OFF + s * C::TILE_BYTES, 16, 1024);
      const uint64_t q_nmaj = smem_desc_sw128(sbase + C::Q_OFF + s * C::TILE_BYTES, C::SLAB_BYTES, 1024);
      const uint64_t do_nmaj = smem_desc_sw128(sbase + C::DO_OFF + s * C::TILE_BYTES, C::SLAB_BYTES, 1024);
      if (!(ok = wait_all(bar_qdo(s), (uint32_t)(it >> 1) & 1u, B_QDO))) break;
      // S^T goes where dQ_{i-1} lies: the rows must have read it out first
      if (it > 0 && !(ok = wait_all(bar_dq_read, ph ^ 1u, B_DQ_READ))) break;
      tc_fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss_elect(tmem_base + C::S_COL, k_kmaj + kmaj_off(kk), q_kmaj + kmaj_off(kk), C::IDESC_S,
                     kk > 0 ? 1u : 0u);
      mma_commit_elect(bar_s);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss_elect(tmem_base + C::DP_COL, v_kmaj + kmaj_off(kk), do_kmaj + kmaj_off(kk), C::IDESC_S,
                     kk > 0 ? 1u : 0u);
      mma_commit_elect(bar_dp);
      if (!(ok = wait_all(bar_ds, ph, B_DS))) break;
      tc_fence_after_sync();
      // dV += P^T dO_i and dK += dS^T Q_i (K = the 128 queries, 16 per MMA step = 8 TMEM
      // columns of bf16 pairs; queries 64-127 start at column 64)
#pragma unroll
      for (int kk = 0; kk < BT / 16; ++kk)
        mma_ts_elect(tmem_base + C::DV_COL, tmem_base + C::S_COL + pcol(kk), do_nmaj + rows16_off(kk), C::IDESC_KV,
                     (it > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
      for (int kk = 0; kk < BT / 16; ++kk)
        mma_ts_elect(tmem_base + C::DK_COL, tmem_base + C::DP_COL + pcol(kk), q_nmaj + rows16_off(kk), C::IDESC_KV,
                     (it > 0 || kk > 0) ? 1u : 0u);
      // dQ_i = dS K_j (K = the 128 keys) into the columns P^T occupied: after the dV MMAs that
      // read it (MMAs of one thread run in order)
#pragma unroll
      for (int kk = 0; kk < BT / 16; ++kk)
        mma_ss_elect(tmem_base + C::S_COL, st_mmaj + rows16_off(kk), k_nmaj + rows16_off(kk), C::IDESC_Q,
                     kk > 0 ? 1u : 0u);
      mma_commit_elect(bar_dq);
      mma_commit_elect(bar_qdo_empty(s));
    }
    // every MMA complete (for the dK / dV epilogue and before TMEM is freed)
    mma_commit_elect(bar_done);
    mbar_wait(bar_done, 0, p.st, nullptr, (K_ATTN_BWD << 8) | B_DONE);
  } else {
    // =================== rows: warps 0-7, thread t = TMEM lane t % 128 ===================
    const int tt = threadIdx.x & (BT - 1);  // key row of the tile (the dQ tile: query row)
    const int half = warp >> 2;             // queries (dQ / dK / dV columns) [64 half, 64 half + 64)
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int key = k0 + tt;
    const bool key_ok = key < p.Nk;
    const float* lse_row = p.lse + (int64_t)bh * p.Nq;
    const float* dsum_row = p.dsum + (int64_t)bh * p.Nq;
    uint8_t* st_row = smem + C::ST_OFF + half * C::SLAB_BYTES + tt * 128;  // key row in slab `half`
    const float4* ld4 = reinterpret_cast<const float4*>(smem + C::LD_OFF);
    float2* ld_mine = reinterpret_cast<float2*>(smem + C::LD_OFF) + tt;
    // this warp's own 32 staging rows: its dS rows, then its 32 x 32 fp32 dQ blocks
    const uint32_t scratch = sbase + C::ST_OFF + half * C::SLAB_BYTES + (warp & 3) * 32 * 128;
    constexpr int DQ_CHUNKS = D / 64;  // 32-column dQ chunks per warp
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int it = 0; ok && it < n_it; ++it) {
      const int i = i_begin + it, q0 = i * BT;
      const uint32_t ph = (uint32_t)it & 1u;
      // every (key, query) pair of the step visible and inside the tensors
      const bool full = (k0 + BT <= p.Nk) && (q0 + BT <= p.Nq) && (!p.causal || i > j);
      // (LSE log2 e, D) of query q0 + t; a row past the end or with no visible key gets
      // +inf, so that exp2(s scale log2 e - inf) = 0 needs no test below
      float2 mine = make_float2(INFINITY, 0.f);
      if (half == 0 && q0 + tt < p.Nq) {
        const float l = lse_row[q0 + tt];
        mine.x = l == -INFINITY ? INFINITY : l * kLog2e;
        mine.y = dsum_row[q0 + tt];
      }
      if (!(ok = wait_all(bar_s, ph, B_S))) break;
      // every row warp is past the previous step's reads of the (LSE, D) block: it arrived on
      // dq_read, which the S MMA of this step waited for
      if (half == 0) *ld_mine = mine;
      // this warp's dQ blocks of the previous step have left the staging rows it rewrites now
      if (lane == 0) bulk_wait_read<0>();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ld);
      if (!(ok = wait_all(bar_ld, ph, B_LD))) break;
      if (!(ok = wait_all(bar_dp, ph, B_DP))) break;
      tc_fence_after_sync();
#pragma unroll 1
      for (int c = 64 * half; c < 64 * half + 64; c += 32) {
        uint32_t sr[32], dr[32];
        tmem_ld32(tmem_base + lane_base + C::S_COL + c, sr);
        tmem_ld32(tmem_base + lane_base + C::DP_COL + c, dr);
        uint32_t pw[16], dw[16];
        if (full)
          bwd_p_ds<false>(sr, dr, ld4 + c / 2, sl2, key, q0 + c, true, false, pw, dw);
        else
          bwd_p_ds<true>(sr, dr, ld4 + c / 2, sl2, key, q0 + c, key_ok, p.causal != 0, pw, dw);
        // P^T / dS^T as bf16 pairs: queries c .. c+31 to columns c/2 (+32 for the second half),
        // all of them already read by this warp and by no other
        const uint32_t oc = c / 2 + (c >= 64 ? 32 : 0);
        tmem_st16(tmem_base + lane_base + C::S_COL + oc, pw);
        tmem_st16(tmem_base + lane_base + C::DP_COL + oc, dw);
        // dS^T row `key`, queries c .. c+31: 16-byte chunks (c % 64) / 8 .. +3 of slab c / 64,
        // chunk q of row r stored at position q ^ (r % 8) (128-byte swizzle)
        const int cq0 = (c % 64) / 8;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          *reinterpret_cast<uint4*>(st_row + (((cq0 + q4) ^ (tt & 7)) * 16)) =
              make_uint4(dw[4 * q4], dw[4 * q4 + 1], dw[4 * q4 + 2], dw[4 * q4 + 3]);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      fence_proxy_async_smem();  // the staged dS is read by the tensor core (async proxy)
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ds);
      // dQ_i = scale dS K_j: thread t holds query row q0 + t % 128.  The warp's columns leave
      // TMEM first (so the next step's S MMA may overwrite them); then per 32 columns the warp
      // stages its 32 x 32 block (swizzled like the map) in its own staging rows, which the dQ
      // MMA has finished reading, and one lane adds it into the accumulator with a TMA
      // reduce-add (rows past Nq are clipped by the map; a block wholly past the end is skipped).
      if (!(ok = wait_all(bar_dq, ph, B_DQ))) break;
      tc_fence_after_sync();
      uint32_t r[DQ_CHUNKS][32];
#pragma unroll
      for (int m = 0; m < DQ_CHUNKS; ++m)
        tmem_ld32(tmem_base + lane_base + C::S_COL + (half * DQ_CHUNKS + m) * 32, r[m]);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_dq_read);
      const bool rows_in = q0 + (warp & 3) * 32 < p.Nq;
      uint8_t* brow = smem + (scratch - sbase) + lane * 128;
#pragma unroll
      for (int m = 0; m < DQ_CHUNKS; ++m) {
        if (m > 0) {  // the previous block has been read out of the staging rows
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
        }
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4)
          *reinterpret_cast<float4*>(brow + ((q4 ^ (lane & 7)) * 16)) =
              make_float4(__uint_as_float(r[m][4 * q4]) * p.scale, __uint_as_float(r[m][4 * q4 + 1]) * p.scale,
                          __uint_as_float(r[m][4 * q4 + 2]) * p.scale, __uint_as_float(r[m][4 * q4 + 3]) * p.scale);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && rows_in) {
          tma_reduce_add_3d(&tm_dq, scratch, (half * DQ_CHUNKS + m) * 32, q0 + (warp & 3) * 32, bh);
          bulk_commit_group();
        }
      }
    }
    // the last dQ blocks: read out of shared memory and added before the CTA may exit
    if (lane == 0) bulk_wait_all();
    __syncwarp();
    // dK_j, dV_j rows (key rows of the tile), columns [half D/2, half D/2 + D/2)
    if (ok && n_it > 0) ok = wait_all(bar_done, 0, B_DONE);
    if (ok) {
      tc_fence_after_sync();
      __nv_bfloat16* dkrow = p.dk + ((int64_t)bh * p.Nk + key) * D;
      __nv_bfloat16* dvrow = p.dv + ((int64_t)bh * p.Nk + key) * D;
#pragma unroll 1
      for (int c = half * (D / 2); c < half * (D / 2) + D / 2; c += 32) {
        uint32_t rk[32], rv[32];
        if (n_it > 0) {
          tmem_ld32(tmem_base + lane_base + C::DK_COL + c, rk);
          tmem_ld32(tmem_base + lane_base + C::DV_COL + c, rv);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) rk[e] = rv[e] = 0u;
        }
        uint4 wk[4], wv[4];
        uint32_t* k32 = reinterpret_cast<uint32_t*>(wk);
        uint32_t* v32 = reinterpret_cast<uint32_t*>(wv);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          k32[e] = pack_bf16x2(__uint_as_float(rk[2 * e]) * p.scale, __uint_as_float(rk[2 * e + 1]) * p.scale);
          v32[e] = pack_bf16x2(__uint_as_float(rv[2 * e]), __uint_as_float(rv[2 * e + 1]));
        }
        if (key_ok) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            reinterpret_cast<uint4*>(dkrow + c)[e] = wk[e];
            reinterpret_cast<uint4*>(dvrow + c)[e] = wv[e];
          }
        }
      }
    }
  }

  // ---- teardown ----
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kBwdMma) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kBwdTmemCols);
  }
}

constexpr int kMaxDevices = 64;

template <int D>
cudaError_t launch_bwd_d(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                         const CUtensorMap& mdo, const CUtensorMap& mdq, const BwdParams& p, cudaStream_t s) {
  static bool attr_set[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(attn_bwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             BwdCfg<D>::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const unsigned grid = (unsigned)p.nkt * (unsigned)p.BH;
  attn_bwd_tc_kernel<D><<<grid, kBwdThreads, BwdCfg<D>::SMEM_BYTES, s>>>(mq, mk, mv, mdo, mdq, p);
  return cudaGetLastError();
}

}  // namespace

size_t attn_bwd_workspace_floats(int B, int H, int Nq, int d) { return (size_t)B * H * Nq * ((size_t)d + 1); }

cudaError_t launch_attn_bwd(const BwdArgs& a, float* workspace, const DevStatus& st, cudaStream_t s,
                            const char** why) {
  const int d = a.d, BH = a.B * a.H;
  const int64_t rb = 2 * (int64_t)d;  // bytes per row
  const int64_t rows = (int64_t)BH * a.Nq;
  float* dq_acc = workspace;
  float* dsum = workspace + rows * d;
  CUtensorMap mq, mk, mv, mdo, mdq;
  if (!make_tile_map(&mq, a.q, d, a.Nq, rb, BH, rb * a.Nq) || !make_tile_map(&mk, a.k, d, a.Nk, rb, BH, rb * a.Nk) ||
      !make_tile_map(&mv, a.v, d, a.Nk, rb, BH, rb * a.Nk) ||
      !make_tile_map(&mdo, a.dout, d, a.Nq, rb, BH, rb * a.Nq) ||
      !make_f32_tile_map(&mdq, dq_acc, d, a.Nq, 2 * rb, BH, 2 * rb * a.Nq, 32)) {
    if (why) *why = "cuTensorMapEncodeTiled failed or is unavailable";
    return cudaErrorInvalidValue;
  }
  bwd_pre_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(static_cast<const __nv_bfloat16*>(a.o),
                                                            static_cast<const __nv_bfloat16*>(a.dout), dsum, dq_acc,
                                                            rows, d);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  BwdParams p;
  p.dq_acc = dq_acc;
  p.lse = a.lse;
  p.dsum = dsum;
  p.dk = static_cast<__nv_bfloat16*>(a.dk);
  p.dv = static_cast<__nv_bfloat16*>(a.dv);
  p.Nq = a.Nq;
  p.Nk = a.Nk;
  p.causal = a.causal;
  p.nkt = (a.Nk + BT - 1) / BT;
  p.nqt = (a.Nq + BT - 1) / BT;
  p.BH = BH;
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.st = st;
  e = d == 128 ? launch_bwd_d<128>(mq, mk, mv, mdo, mdq, p, s) : launch_bwd_d<64>(mq, mk, mv, mdo, mdq, p, s);
  if (e != cudaSuccess) return e;
  const int64_t n = rows * d;
  bwd_post_kernel<<<(unsigned)((n / 4 + 255) / 256), 256, 0, s>>>(dq_acc, static_cast<__nv_bfloat16*>(a.dq), n);
  return cudaGetLastError();
}

}  // namespace oa
