// attn_bwd.cu -- attention backward on the 5th-generation tensor cores (tcgen05, tensor
// memory, TMA), bf16 inputs, fp32 accumulation, d = 64 / 128.
//
// What it computes: the gradients of O = softmax(scale Q K^T) V for a given dO, with the
// attention weights recomputed from the scores and the forward's per-row LSE instead of
// being read back from a stored [N, N] matrix (page "Online softmax in attention -- why
// and how", "Where this is heading: FA2": on backward, recompute the scores from the cached
// softmax statistics).  With P = exp(scale S - LSE) (S = Q K^T, masked keys 0):
//   dV = P^T dO,   dP = dO V^T,   D = rowsum(dO o O),   dS = P o (dP - D),
//   dQ = scale dS K,   dK = scale dS^T Q    (the kernels carry scale dS, formed with one FMA).
//
// Three launches: a pre-pass (D per query row; the fp32 dQ accumulator zeroed), the main
// kernel (attn_bwd_tc_kernel at d = 128, described here; attn_bwd_tc64_kernel at d = 64, the
// same roles pipelined one step deeper, described at its definition), and a post-pass (dQ to
// bf16).  Main kernel, key-tile outer: one CTA per (b, h, 128 keys); K_j and V_j stay in shared
// memory while the query tiles i that see any of its keys stream through a 2-stage TMA ring with
// their dO tiles (causal: query i sees keys j <= i + Nk - Nq, the queries being the sequence's last
// Nq positions; per sequence for packed sequences).  Per query tile:
//   S^T  = K_j Q_i^T,   dP^T = V_j dO_i^T           (SS MMAs into TMEM, lanes = keys, N = 128)
//   P^T  elementwise as soon as S^T is in, while dP^T computes (P^T as bf16 back into TMEM)
//   dV_j += P^T dO_i                                 (TS MMA: A from TMEM), while the rows
//   dS^T elementwise from dP^T and the P^T kept in registers (bf16 into TMEM and shared memory)
//   dK_j += dS^T Q_i                                 (TS MMA, accumulates in TMEM)
//   dQ_i  = dS K_j                                   (SS MMA: A = the staged dS, read M-major)
// and the dQ_i tile is added into the fp32 accumulator in global memory (the tiles of
// other key blocks add into the same rows) by TMA reduce-adds of 32 x 32 blocks staged in
// shared memory.  dK_j, dV_j leave TMEM once, at the end.  The 128 (LSE log2 e, D) pairs
// of a query tile are loaded once per step into shared memory and read as broadcasts.
//
// GB300 mapping (352 threads, one CTA per SM):
//   warps 0-7  warp w reaches TMEM lanes 32 (w % 4) .. +31, so thread t owns key row t % 128
//              of the tile for the elementwise passes and the dK/dV epilogue, and query row
//              t % 128 of the dQ tile; warps 0-3 take queries (or columns) [0, 64), warps 4-7
//              [64, 128): two row warps per SM sub-partition
//   warp 8     TMA producer (K_j, V_j once; Q_i, dO_i per step)
//   warp 9     MMA issue (whole warp, one elected lane); owns the TMEM allocation
//   warp 10    dQ reducer: issues the TMA reduce-adds of the staged dQ blocks
// TMEM (512 columns): S^T [0, 128) -> P^T bf16 (queries 0-63 in [0, 32), 64-127 in [64, 96):
// each warp overwrites only scores it has read); dP^T [128, 256) -> dS^T bf16 likewise at +128
// -> dQ_i fp32 [128, 128 + d), written after the dK MMAs have read dS^T, so that the next
// step's S^T MMAs need not wait for the dQ read-out (only its dP^T MMAs do); dV [256, 256 + d);
// dK [256 + d, 256 + 2d).
//
// Every wait is bounded (oa_common.cuh); a wait that expires aborts the CTA, which falls
// through to its teardown with TMEM freed.
#include "oa_internal.h"

namespace oa {
namespace {

constexpr int BT = 128;                  // keys per CTA tile = query rows per step
constexpr int kBwdRowWarps = 8;
constexpr int kBwdThreads = 32 * (kBwdRowWarps + 3);
constexpr int kBwdProducer = kBwdRowWarps;
constexpr int kBwdMma = kBwdRowWarps + 1;
constexpr int kBwdReducer = kBwdRowWarps + 2;
constexpr uint32_t kBwdTmemCols = 512;
// Key/value planes per dispatch group: the CTAs of kBwdPlaneGroup planes come before those of the
// next planes, so the dQ accumulator rows and the Q / dO tiles that the running CTAs share stay in
// L2 (key tile order over all planes at once spreads them over every head's rows).
constexpr int kBwdPlaneGroup = 4;

template <int D>
struct BwdCfg {
  static constexpr int SLABS = D / 64;        // 128-byte swizzle atoms along d
  static constexpr int DQ_CHUNKS = D / 64;    // 32-column dQ chunks per row warp
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
  // -LSE log2 e of the step's 128 query rows, then -D scale (-inf / 0 past the end)
  static constexpr int LD_OFF = ST_OFF + ST_BYTES;
  static constexpr int BAR_OFF = LD_OFF + BT * 8;
  // kv_full, q_full[2], q_empty[2], s_full[2], dp_full[2], ds_ready[2], dq_full, dq_read, done,
  // ld_ready[2], dq_staged[2], p_ready[2], do_full[2], do_empty[2], dq_staged_hi[2] ([s]: ring stage
  // s; [h]: the query half h = queries 64h .. 64h + 63 of the step; s_full and dp_full complete
  // together for both halves)
  static constexpr int NUM_BARS = 26;
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;  // + slack to align the base to 1024
  static constexpr uint32_t S_COL = 0, DP_COL = 128, DV_COL = 256, DK_COL = 256 + D;
  // S^T = K Q^T and dP^T = V dO^T for the 128 queries: both operands K-major
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
  int Nq, Nk, causal, nkt, nqt;  // dense: lengths and tiles; packed: the longest key sequence's tiles (nkt)
  int BHkv;   // dense: key/value planes (B * H_kv); packed: sequences * H_kv.  The grid covers nkt key
              // tiles of each
  int group;  // query heads per key/value head (H / H_kv)
  int H, Hkv;                       // packed: head counts of the token-major rows
  const int32_t *cu_q, *cu_k;       // packed: sequence offsets [num_seqs + 1] (NULL: dense)
  int total_q, total_k;             // packed: tokens in the Q / K tensors
  float scale, scale_log2;
  int64_t lse_elems, dk_elems;  // extents of lse / dsum and of dk / dv (the debug build's checks)
  DevStatus st;
};

enum BwdWait : unsigned { B_KV = 1, B_QDO, B_QDO_EMPTY, B_S, B_DP, B_DS, B_DQ, B_DQ_READ, B_DONE, B_LD, B_DQ_STAGED };

// Shared-memory offset of the 32 x 32 fp32 dQ block (row warp w, chunk m) of a step: 4 KB each,
// in that step's Q stage and then its dO stage (8 warps x DQ_CHUNKS x 4 KB = the two tiles),
// which no MMA reads once the step's dQ MMA is complete.
template <class C>
__device__ __forceinline__ uint32_t bwd_dq_block(uint32_t q_stage_off, int w, int m) {
  const uint32_t off = (uint32_t)((w * C::DQ_CHUNKS + m) * 4096);
  return q_stage_off + (off < (uint32_t)C::TILE_BYTES ? off : off - C::TILE_BYTES + (C::DO_OFF - C::Q_OFF));
}

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

// P^T for 64 queries q_first .. q_first + 63 of one key row: sr the fp32 S^T columns, nl the
// negated LSE log2 e of those queries (four per float4).  pp keeps P^T in fp32 pairs for the dS^T
// pass, pw the bf16 pairs that the dV MMA reads.  MASK applies the key and causal tests as an
// exponent of -inf (no branch); `key` is the key's index minus the causal offset, so the causal test
// is key <= q.
template <bool MASK>
__device__ __forceinline__ void bwd_p(const uint32_t (&sr)[64], const float4* nl, uint64_t sl2x2, int key, int q_first,
                                      bool key_ok, bool causal, uint64_t (&pp)[32], uint32_t (&pw)[32]) {
#pragma unroll
  for (int e = 0; e < 64; e += 4) {
    const ulonglong2 nlv = *reinterpret_cast<const ulonglong2*>(nl + e / 4);
#pragma unroll
    for (int h = 0; h < 4; h += 2) {
      const uint64_t a = f2_fma(f2_pack(__uint_as_float(sr[e + h]), __uint_as_float(sr[e + h + 1])), sl2x2,
                                h ? nlv.y : nlv.x);
      float a0, a1;
      f2_unpack(a, a0, a1);
      if (MASK) {
        const int q = q_first + e + h;
        a0 = (key_ok && (!causal || key <= q)) ? a0 : -INFINITY;
        a1 = (key_ok && (!causal || key <= q + 1)) ? a1 : -INFINITY;
      }
      const float p0 = ex2(a0), p1 = ex2(a1);
      pp[(e + h) / 2] = f2_pack(p0, p1);
      pw[(e + h) / 2] = pack_bf16x2(p0, p1);
    }
  }
}
// scale dS^T = P^T (dP^T scale - D scale) for the same 64 queries, one FMA per pair: dr the fp32 dP^T
// columns, nd the negated D scale of those queries, s2x2 the scale twice, pp the fp32 P^T of bwd_p;
// dw the bf16 pairs.  With the scale inside dS, dQ = dS K and dK = dS^T Q need no further scaling.
__device__ __forceinline__ void bwd_ds(const uint32_t (&dr)[64], const float4* nd, uint64_t s2x2, const uint64_t (&pp)[32],
                                       uint32_t (&dw)[32]) {
#pragma unroll
  for (int e = 0; e < 64; e += 4) {
    const ulonglong2 ndv = *reinterpret_cast<const ulonglong2*>(nd + e / 4);
#pragma unroll
    for (int h = 0; h < 4; h += 2) {
      const uint64_t dpd = f2_fma(f2_pack(__uint_as_float(dr[e + h]), __uint_as_float(dr[e + h + 1])), s2x2,
                                  h ? ndv.y : ndv.x);
      const uint64_t ds = f2_mul(pp[(e + h) / 2], dpd);
      float d0, d1;
      f2_unpack(ds, d0, d1);
      dw[(e + h) / 2] = pack_bf16x2(d0, d1);
    }
  }
}

// The CTA's geometry.  Rows: Q / dO / dQ row of query q is qrow0 + q, K / V / dK / dV row of key
// k is krow0 + k (TMA coordinates); query head t of the group is TMA plane qplane0 + t; the LSE / D
// entry of (q, t) is lbase + q lq + t lt; the dK / dV row of key k starts at (dkbase + k dks) d.
struct BwdGeom {
  int j, k0;  // key tile and its first key
  int Nq, Nk, nqt, qrow0, krow0, qplane0, kplane;
  int off;      // causal: query q sees key k iff k <= q + off (keys minus queries)
  int64_t lbase, lq, lt, dkbase, dks;
  int i_begin;  // first query tile that sees a key of tile j (causal: the one holding query k0 - off)
  int n_it;     // steps: every visible query tile of every query head of the group, head by head
};

// grid.x = nkt * BHkv CTAs in groups of kBwdPlaneGroup key/value planes (the last group may be
// smaller); inside a group the key tile j is the slow index (low j first: for causal those have
// the most query tiles) and the plane the fast one.  A plane is -- dense: (b, key/value head);
// PACKED: (sequence, key/value head) of token-major [tokens, heads, d] tensors, whose sequence s
// owns rows [cu[s], cu[s+1]) (a CTA past its sequence's keys exits at once).
// Returns false for a CTA with nothing to do (its key tile starts past its packed sequence's keys).
template <bool PACKED>
__device__ __forceinline__ bool bwd_geometry(const BwdParams& p, BwdGeom& g) {
  const int g0 = (int)(blockIdx.x / (unsigned)(kBwdPlaneGroup * p.nkt)) * kBwdPlaneGroup;  // first plane
  const int gsz = min(kBwdPlaneGroup, p.BHkv - g0);
  const int g_local = (int)blockIdx.x - g0 * p.nkt;
  g.j = g_local / gsz;
  const int plane = g0 + g_local % gsz;
  g.k0 = g.j * BT;
  if constexpr (PACKED) {
    const int seq = plane / p.Hkv, hkv = plane % p.Hkv;
    const int qb = min(max(p.cu_q[seq], 0), p.total_q), qe = min(max(p.cu_q[seq + 1], qb), p.total_q);
    const int kb = min(max(p.cu_k[seq], 0), p.total_k), ke = min(max(p.cu_k[seq + 1], kb), p.total_k);
    g.Nq = qe - qb;
    g.Nk = ke - kb;
    // a key sequence longer than the grid covers: its tail gets no gradient; report it
    if (g.j == p.nkt - 1 && hkv == 0 && threadIdx.x == 0 && g.Nk > p.nkt * BT)
      record_failure(p.st, kSiteBwdBadSeqlen);
    if (g.k0 >= g.Nk) return false;  // uniform over the CTA; nothing set up yet
    g.qrow0 = qb;
    g.krow0 = kb;
    g.qplane0 = hkv * p.group;
    g.kplane = hkv;
    g.lbase = (int64_t)qb * p.H + (int64_t)hkv * p.group;
    g.lq = p.H;
    g.lt = 1;
    g.dkbase = (int64_t)kb * p.Hkv + hkv;
    g.dks = p.Hkv;
  } else {
    const int kvp = plane;  // (b, key/value head)
    g.Nq = p.Nq;
    g.Nk = p.Nk;
    g.qrow0 = g.krow0 = 0;
    g.qplane0 = kvp * p.group;
    g.kplane = kvp;
    g.lbase = (int64_t)kvp * p.group * p.Nq;
    g.lq = 1;
    g.lt = p.Nq;
    g.dkbase = (int64_t)kvp * p.Nk;
    g.dks = 1;
  }
  g.nqt = (g.Nq + BT - 1) / BT;
  g.off = g.Nk - g.Nq;
  g.i_begin = (p.causal && g.k0 - g.off > 0) ? (g.k0 - g.off) / BT : 0;
  g.n_it = p.group * max(g.nqt - g.i_begin, 0);
  return true;
}

// (query head t of the group, query tile i) of a step; next() steps to the following one without a
// division: query tiles i_begin .. nqt - 1 of head t, then of head t + 1
struct StepPos {
  int t, i;
  __device__ __forceinline__ StepPos next(const BwdGeom& g) const {
    StepPos n{t, i + 1};
    if (n.i == g.nqt) {
      n.i = g.i_begin;
      ++n.t;
    }
    return n;
  }
};

// dK and dV of key row `key` as bf16, columns [half d/2, half d/2 + d/2), from the
// accumulators at TMEM columns dk_col and dv_col of this thread's lane (tl = TMEM base + the warp's
// lane quarter); zeros when the CTA had no step; no store for a key past the end.
template <int D>
__device__ __forceinline__ void bwd_store_dkdv(const BwdParams& p, const BwdGeom& g, uint32_t tl, uint32_t dk_col,
                                               uint32_t dv_col, int half, int key, bool key_ok, bool any_step) {
  __nv_bfloat16* dkrow = p.dk + (g.dkbase + (int64_t)key * g.dks) * D;
  __nv_bfloat16* dvrow = p.dv + (g.dkbase + (int64_t)key * g.dks) * D;
#pragma unroll 1
  for (int c = half * (D / 2); c < half * (D / 2) + D / 2; c += 32) {
    uint32_t rk[32], rv[32];
    if (any_step) {
      tmem_ld32(tl + dk_col + c, rk);
      tmem_ld32(tl + dv_col + c, rv);
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) rk[e] = rv[e] = 0u;
    }
    uint4 wk[4], wv[4];
    uint32_t* k32 = reinterpret_cast<uint32_t*>(wk);
    uint32_t* v32 = reinterpret_cast<uint32_t*>(wv);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      k32[e] = pack_bf16x2(__uint_as_float(rk[2 * e]), __uint_as_float(rk[2 * e + 1]));
      v32[e] = pack_bf16x2(__uint_as_float(rv[2 * e]), __uint_as_float(rv[2 * e + 1]));
    }
    if (key_ok && OA_DCHECK(p.st, (g.dkbase + (int64_t)key * g.dks) * D + c + 32 <= p.dk_elems,
                            (K_ATTN_BWD << 8) | kSiteDebugBase)) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        reinterpret_cast<uint4*>(dkrow + c)[e] = wk[e];
        reinterpret_cast<uint4*>(dvrow + c)[e] = wv[e];
      }
    }
  }
}

template <int D, bool PACKED>
__global__ void __launch_bounds__(kBwdThreads)
    attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  static_assert(D == 128, "d = 64 runs attn_bwd_tc64_kernel");
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_addr(smem_raw);
  const uint32_t pad = (1024u - (raw_s & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_s + pad;

  const uint32_t bar0 = sbase + C::BAR_OFF;
  const uint32_t bar_kv = bar0;
  auto bar_qdo = [&](int s) { return bar0 + 8u * (1 + s); };  // Q_i of stage s landed
  // the Q buffer of stage s free again: its MMAs are complete and the dQ blocks that warps 0-3
  // staged in it have been read by their TMA reduce-adds (the reducer warp); bar_do_empty the same
  // for the dO buffer and warps 4-7.  The reducer adds the Q buffer's blocks first, so the next
  // Q (needed first, by the S MMAs) can load while the dO buffer's blocks are still being read.
  auto bar_qdo_empty = [&](int s) { return bar0 + 8u * (3 + s); };
  auto bar_s = [&](int h) { return bar0 + 8u * (5 + h); };    // S^T (waited on by the rows of half h)
  auto bar_dp = [&](int h) { return bar0 + 8u * (7 + h); };   // dP^T (likewise)
  auto bar_ds = [&](int h) { return bar0 + 8u * (9 + h); };   // P^T, dS^T of half h in TMEM, dS staged
  const uint32_t bar_dq = bar0 + 8u * 11;                     // dQ_i in TMEM
  const uint32_t bar_dq_read = bar0 + 8u * 12;                // dQ_i read out of TMEM (8 warps)
  const uint32_t bar_done = bar0 + 8u * 13;                   // every MMA of the CTA complete
  auto bar_ld = [&](int h) { return bar0 + 8u * (14 + h); };  // half h's (LSE, D) entries written
  // the dQ blocks of the step using stage s are staged in it (8 warps)
  auto bar_dq_staged = [&](int s) { return bar0 + 8u * (16 + s); };  // warps 0-3 staged (Q buffer)
  auto bar_do = [&](int s) { return bar0 + 8u * (20 + s); };             // dO_i of stage s landed
  auto bar_do_empty = [&](int s) { return bar0 + 8u * (22 + s); };
  auto bar_dq_staged_hi = [&](int s) { return bar0 + 8u * (24 + s); };  // warps 4-7 staged (dO buffer)
  auto bar_p = [&](int h) { return bar0 + 8u * (18 + h); };   // P^T of half h in TMEM (4 warps)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  BwdGeom g;
  if (!bwd_geometry<PACKED>(p, g)) return;
  const int k0 = g.k0, Nq = g.Nq, Nk = g.Nk, qrow0 = g.qrow0, qplane0 = g.qplane0, n_it = g.n_it;
  const int64_t lbase = g.lbase, lq = g.lq, lt = g.lt;
  auto next_pos = [&](StepPos sp) { return sp.next(g); };
  const StepPos first_pos{0, g.i_begin};

  if (threadIdx.x == 0) {
    mbar_init(bar_kv, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_qdo(s), 1);
      mbar_init(bar_qdo_empty(s), 1);
      mbar_init(bar_dq_staged(s), kBwdRowWarps / 2);
      mbar_init(bar_dq_staged_hi(s), kBwdRowWarps / 2);
      mbar_init(bar_do(s), 1);
      mbar_init(bar_do_empty(s), 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(bar_s(h), 1);
      mbar_init(bar_dp(h), 1);
      mbar_init(bar_ds(h), kBwdRowWarps / 2);
      mbar_init(bar_p(h), kBwdRowWarps / 2);
      mbar_init(bar_ld(h), kBwdRowWarps / 2);
    }
    mbar_init(bar_dq, 1);
    mbar_init(bar_dq_read, kBwdRowWarps);
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
      tma_load_3d_elect(sbase + C::K_OFF + c * C::SLAB_BYTES, &tm_k, bar_kv, c * 64, g.krow0 + k0, g.kplane);
      tma_load_3d_elect(sbase + C::V_OFF + c * C::SLAB_BYTES, &tm_v, bar_kv, c * 64, g.krow0 + k0, g.kplane);
    }
    int issued_q = 0, issued_do = 0;
    StepPos pos = first_pos;
    for (int it = 0; it < n_it; ++it, pos = next_pos(pos)) {
      const int s = it & 1, q0 = pos.i * BT, qp = qplane0 + pos.t, qy = qrow0 + q0;
      // stage s was last used by step it - 2: Q first (the S MMAs read it first), then dO
      const uint32_t par = (uint32_t)((it >> 1) - 1) & 1u;
      if (it >= 2 && !(ok = wait_all(bar_qdo_empty(s), par, B_QDO_EMPTY))) break;
      mbar_arrive_expect_tx_elect(bar_qdo(s), C::TILE_BYTES);
      for (int c = 0; c < C::SLABS; ++c)
        tma_load_3d_elect(sbase + C::Q_OFF + s * C::TILE_BYTES + c * C::SLAB_BYTES, &tm_q, bar_qdo(s), c * 64, qy,
                          qp);
      ++issued_q;
      if (it >= 2 && !(ok = wait_all(bar_do_empty(s), par, B_QDO_EMPTY))) break;
      mbar_arrive_expect_tx_elect(bar_do(s), C::TILE_BYTES);
      for (int c = 0; c < C::SLABS; ++c)
        tma_load_3d_elect(sbase + C::DO_OFF + s * C::TILE_BYTES + c * C::SLAB_BYTES, &tm_do, bar_do(s), c * 64,
                          qy, qp);
      ++issued_do;
    }
    // drain: every load issued must have landed before the CTA can exit
    for (int it = max(0, issued_q - 2); it < issued_q; ++it)
      mbar_wait(bar_qdo(it & 1), (uint32_t)(it >> 1) & 1u, p.st, nullptr, (K_ATTN_BWD << 8) | B_DONE);
    for (int it = max(0, issued_do - 2); it < issued_do; ++it)
      mbar_wait(bar_do(it & 1), (uint32_t)(it >> 1) & 1u, p.st, nullptr, (K_ATTN_BWD << 8) | B_DONE);
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
      tc_fence_after_sync();
      // S^T into columns that nothing reads any more (the previous step's P^T was read by its dV
      // MMAs, issued earlier); dP^T into the columns of the previous step's dQ, once the rows have
      // read it out
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss_elect(tmem_base + C::S_COL, k_kmaj + kmaj_off(kk), q_kmaj + kmaj_off(kk), C::IDESC_S, kk > 0 ? 1u : 0u);
      mma_commit_elect(bar_s(0));
      mma_commit_elect(bar_s(1));
      if (it > 0 && !(ok = wait_all(bar_dq_read, ph ^ 1u, B_DQ_READ))) break;
      if (!(ok = wait_all(bar_do(s), (uint32_t)(it >> 1) & 1u, B_QDO))) break;  // dO_i landed
      tc_fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ss_elect(tmem_base + C::DP_COL, v_kmaj + kmaj_off(kk), do_kmaj + kmaj_off(kk), C::IDESC_S, kk > 0 ? 1u : 0u);
      mma_commit_elect(bar_dp(0));
      mma_commit_elect(bar_dp(1));
      // dV += P^T dO_i half by half as the rows write P^T (K = 16 queries per MMA step = 8 TMEM
      // columns of bf16 pairs; queries 64-127 start at column 64), while dP^T computes; then
      // dK += dS^T Q_i likewise
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (!(ok = wait_all(bar_p(h), ph, B_DS))) break;
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 4 * h; kk < 4 * h + 4; ++kk)
          mma_ts_elect(tmem_base + C::DV_COL, tmem_base + C::S_COL + pcol(kk), do_nmaj + rows16_off(kk),
                       C::IDESC_KV, (it > 0 || kk > 0) ? 1u : 0u);
      }
      if (!ok) break;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (!(ok = wait_all(bar_ds(h), ph, B_DS))) break;
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 4 * h; kk < 4 * h + 4; ++kk)
          mma_ts_elect(tmem_base + C::DK_COL, tmem_base + C::DP_COL + pcol(kk), q_nmaj + rows16_off(kk),
                       C::IDESC_KV, (it > 0 || kk > 0) ? 1u : 0u);
      }
      if (!ok) break;
      // dQ_i = dS K_j (K = the 128 keys) into the columns dS^T occupied: after the dK MMAs that
      // read it (MMAs of one thread run in order)
#pragma unroll
      for (int kk = 0; kk < BT / 16; ++kk)
        mma_ss_elect(tmem_base + C::DP_COL, st_mmaj + rows16_off(kk), k_nmaj + rows16_off(kk), C::IDESC_Q,
                     kk > 0 ? 1u : 0u);
      mma_commit_elect(bar_dq);
    }
    // every MMA complete (for the dK / dV epilogue and before TMEM is freed)
    mma_commit_elect(bar_done);
    mbar_wait(bar_done, 0, p.st, nullptr, (K_ATTN_BWD << 8) | B_DONE);
  } else if (warp == kBwdReducer) {
    // ============ dQ reducer (whole warp, one lane issues): TMA reduce-adds of the blocks ============
    // Step `it` uses stage it & 1 for Q_i, dO_i and then for the row warps' dQ blocks; each block
    // is added into rows q0 + 32 (w % 4) .. + 31 (clipped at Nq; skipped when wholly past it)
    // and columns 32 (DQ_CHUNKS (w / 4) + m) of the fp32 accumulator.
    bool ok = true;
    StepPos pos = first_pos;
    for (int it = 0; ok && it < n_it; ++it, pos = next_pos(pos)) {
      const int s = it & 1, q0 = pos.i * BT, qp = qplane0 + pos.t, qy = qrow0 + q0;
      const uint32_t stage_base = C::Q_OFF + (uint32_t)s * C::TILE_BYTES;
      const uint32_t par = (uint32_t)(it >> 1) & 1u;
      // warps 0-3 staged their blocks in the Q buffer, warps 4-7 in the dO buffer: one commit
      // group each, the Q buffer's first
      for (int hw = 0; hw < 2 && ok; ++hw) {
        if (!(ok = wait_all(hw ? bar_dq_staged_hi(s) : bar_dq_staged(s), par, B_DQ_STAGED))) break;
        if (lane == 0) {
          for (int w = 4 * hw; w < 4 * hw + 4; ++w) {
            if (q0 + (w & 3) * 32 >= Nq) continue;
            for (int m = 0; m < C::DQ_CHUNKS; ++m)
              tma_reduce_add_3d(&tm_dq, sbase + bwd_dq_block<C>(stage_base, w, m),
                                ((w >> 2) * C::DQ_CHUNKS + m) * 32, qy + (w & 3) * 32, qp);
          }
          bulk_commit_group();
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) bulk_wait_read<1>();  // the Q buffer's blocks have been read: refill it
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_qdo_empty(s));
      if (lane == 0) bulk_wait_read<0>();  // and the dO buffer's
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_do_empty(s));
    }
    if (lane == 0) bulk_wait_all();  // every add performed before the CTA exits
    __syncwarp();
  } else {
    // =================== rows: warps 0-7, thread t = TMEM lane t % 128 ===================
    const int tt = threadIdx.x & (BT - 1);  // key row of the tile (the dQ tile: query row)
    const int half = warp >> 2;             // queries (dQ / dK / dV columns) [64 half, 64 half + 64)
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int key = k0 + tt;
    const bool key_ok = key < Nk;

    uint8_t* st_row = smem + C::ST_OFF + half * C::SLAB_BYTES + tt * 128;  // key row in slab `half`
    const float4* nl4 = reinterpret_cast<const float4*>(smem + C::LD_OFF);
    const float4* nd4 = reinterpret_cast<const float4*>(smem + C::LD_OFF + BT * 4);
    // threads 0-63 of each half own the (LSE, D) entries of that half's queries
    const int ld_q = 64 * half + tt;
    float* nl_mine = reinterpret_cast<float*>(smem + C::LD_OFF) + ld_q;
    float* nd_mine = reinterpret_cast<float*>(smem + C::LD_OFF + BT * 4) + ld_q;
    constexpr int DQ_CHUNKS = C::DQ_CHUNKS;
    const uint64_t sl2x2 = f2_pack(p.scale_log2, p.scale_log2);
    const uint64_t sl2 = f2_pack(p.scale, p.scale);
    // (LSE, D) of query q0 + ld_q of step `step`, as loaded values (converted when stored)
    auto load_ld = [&](int step, StepPos sp, float& l, float& dd) {
      l = -INFINITY;
      dd = 0.f;
      const int q = sp.i * BT + ld_q;
      if (tt < 64 && step < n_it && q < Nq) {
        const int64_t row = lbase + (int64_t)q * lq + (int64_t)sp.t * lt;
        if (OA_DCHECK(p.st, row < p.lse_elems, (K_ATTN_BWD << 8) | (kSiteDebugBase + 1))) {
          l = p.lse[row];
          dd = p.dsum[row];
        }
      }
    };
    // issued one step ahead: the loads' latency hides behind the step's dV / dK / dQ MMAs
    float next_l, next_d;
    load_ld(0, first_pos, next_l, next_d);
    bool ok = true;
    StepPos pos = first_pos;
    for (int it = 0; ok && it < n_it; ++it) {
      const int i = pos.i, q0 = i * BT;
      const uint32_t ph = (uint32_t)it & 1u;
      // every (key, query) pair of the step visible and inside the tensors
      const bool full = (k0 + BT <= Nk) && (q0 + BT <= Nq) && (!p.causal || k0 + BT - 1 <= q0 + g.off);
      if (!(ok = wait_all(bar_s(half), ph, B_S))) break;
      // -LSE log2 e and -D scale of query q0 + ld_q; a row past the end or with no visible key gets
      // -inf, so that exp2(s scale log2 e - inf) = 0 needs no test below
      // every row warp is past the previous step's reads of the (LSE, D) block: this warp waited
      // for that step's dQ MMA, issued only after all eight warps had arrived on ds_ready
      if (tt < 64) {
        *nl_mine = next_l == -INFINITY ? -INFINITY : -next_l * kLog2e;
        *nd_mine = -next_d * p.scale;
      }
      if (lane == 0) mbar_arrive(bar_ld(half));
      if (!(ok = wait_all(bar_ld(half), ph, B_LD))) break;
      tc_fence_after_sync();
      // this warp's 64 columns of S^T (then of dP^T); P^T and dS^T go as bf16 pairs into the first
      // 32 of them, which this warp has read and no other warp touches
      const uint32_t sc = tmem_base + lane_base + C::S_COL + 64 * half;
      const uint32_t dc = tmem_base + lane_base + C::DP_COL + 64 * half;
      uint64_t pp[32];  // P^T of the 64 queries in fp32, for the dS^T pass
      {
        uint32_t sr[64], pw[32];
        tmem_ld32x2(sc, sc + 32, sr);
        if (full)
          bwd_p<false>(sr, nl4 + 16 * half, sl2x2, key, q0 + 64 * half, true, false, pp, pw);
        else
          bwd_p<true>(sr, nl4 + 16 * half, sl2x2, key - g.off, q0 + 64 * half, key_ok, p.causal != 0, pp, pw);
        tmem_st32(sc, pw);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p(half));
      if (!(ok = wait_all(bar_dp(half), ph, B_DP))) break;
      tc_fence_after_sync();
      {
        uint32_t dr[64], dw[32];
        tmem_ld32x2(dc, dc + 32, dr);
        bwd_ds(dr, nd4 + 16 * half, sl2, pp, dw);
        tmem_st32(dc, dw);
        // dS^T row `key`, queries 64 half .. +63: the 128-byte row of slab `half`, 16-byte chunk q
        // stored at position q ^ (row % 8) (128-byte swizzle)
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8)
          *reinterpret_cast<uint4*>(st_row + ((q8 ^ (tt & 7)) * 16)) =
              make_uint4(dw[4 * q8], dw[4 * q8 + 1], dw[4 * q8 + 2], dw[4 * q8 + 3]);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      fence_proxy_async_smem();  // the staged dS is read by the tensor core (async proxy)
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ds(half));
      pos = next_pos(pos);  // the next step's (head, tile); its (LSE, D) load is issued now
      load_ld(it + 1, pos, next_l, next_d);
      // dQ_i = (scale dS) K_j: thread t holds query row q0 + t % 128.  The warp's columns leave
      // TMEM first (so the next step's dP MMA may overwrite them); then per 32 columns the warp
      // stages its 32 x 32 block (swizzled like the map) in its own staging rows, which the dQ
      // MMA has finished reading, and one lane adds it into the accumulator with a TMA
      // reduce-add (rows past Nq are clipped by the map; a block wholly past the end is skipped).
      if (!(ok = wait_all(bar_dq, ph, B_DQ))) break;
      tc_fence_after_sync();
      uint32_t r[DQ_CHUNKS * 32];  // this warp's 64 dQ columns, one wait
      const uint32_t a0 = tmem_base + lane_base + C::DP_COL + half * 64;
      tmem_ld32x2(a0, a0 + 32, r);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_dq_read);
      const uint32_t stage_base = C::Q_OFF + (uint32_t)(it & 1) * C::TILE_BYTES;  // this step's Q stage
#pragma unroll
      for (int m = 0; m < DQ_CHUNKS; ++m) {
        uint8_t* brow = smem + bwd_dq_block<C>(stage_base, warp, m) + lane * 128;
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4)
          *reinterpret_cast<float4*>(brow + ((q4 ^ (lane & 7)) * 16)) =
              make_float4(__uint_as_float(r[32 * m + 4 * q4]), __uint_as_float(r[32 * m + 4 * q4 + 1]),
                          __uint_as_float(r[32 * m + 4 * q4 + 2]), __uint_as_float(r[32 * m + 4 * q4 + 3]));
      }
      fence_proxy_async_smem();  // the blocks are read by the reducer warp's TMA (async proxy)
      __syncwarp();
      if (lane == 0) mbar_arrive(warp < 4 ? bar_dq_staged(it & 1) : bar_dq_staged_hi(it & 1));
    }
    // dK_j, dV_j rows (key rows of the tile), columns [half D/2, half D/2 + D/2)
    if (ok && n_it > 0) ok = wait_all(bar_done, 0, B_DONE);
    if (ok) {
      tc_fence_after_sync();
      bwd_store_dkdv<D>(p, g, tmem_base + lane_base, C::DK_COL, C::DV_COL, half, key, key_ok, n_it > 0);
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

// ---------------------------------------------------------------------------------------------
// d = 64: a deeper pipeline across steps.  At d = 64 TMEM has columns to spare (S^T 128 + dP^T 128
// + dV 64 + dK 64 = 384 of 512) and shared memory has room (the K, V, Q, dO tiles are half the
// size), so dQ gets TMEM columns and a staging buffer of its own, and Q / dO a third ring stage.
// Then the next step's S^T MMAs are issued right after this step's dV MMAs, and the row warps
// read out and stage the previous step's dQ between their P and dS passes instead of waiting for
// this step's dK and dQ MMAs:
//   MMA warp:   dV_n, S_{n+1}, dK_n, dQ_n (once dQ_{n-1} has been read out), dP_{n+1}
//   row warps:  P pass n, dQ_{n-1} read-out and staging, dS pass n, (LSE, D) of step n + 1
// The last 64 TMEM columns hold K and V (bf16 pairs, copied in by the row warps once per CTA), so the
// S^T = K Q^T and dP^T = V dO^T MMAs take their A operand from TMEM: the two 16 KB tiles are not
// re-read from shared memory every step, whose bandwidth the tensor core's operand reads and the row
// warps' accesses otherwise share.  The (LSE, D) entries of a step are double-buffered, so the row
// warps write the next step's entries as soon as their own dS pass is done.
// Everything else (roles, passes, masks, the dQ reduce-adds, the dK / dV epilogue) is as in
// attn_bwd_tc_kernel.
// ---------------------------------------------------------------------------------------------
struct Bwd64Cfg {
  static constexpr int D = 64;
  static constexpr int TILE_BYTES = BT * 128;  // 128 rows x 64 bf16: one 128-byte swizzle slab
  static constexpr int NST = 3;                // Q / dO ring stages
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + TILE_BYTES;
  static constexpr int Q_OFF = V_OFF + TILE_BYTES;
  static constexpr int DO_OFF = Q_OFF + NST * TILE_BYTES;
  static constexpr int ST_OFF = DO_OFF + NST * TILE_BYTES;  // dS of a step: two 64-query slabs
  static constexpr int DQB_OFF = ST_OFF + 2 * TILE_BYTES;   // dQ staging: warp w's 32 x 32 fp32 block at w * 4 KB
  // two buffers (step parity) of the step's 128 (-LSE log2 e) then 128 (-D scale)
  static constexpr int LD_OFF = DQB_OFF + kBwdRowWarps * 4096;
  static constexpr int LD_BYTES = BT * 8;
  static constexpr int BAR_OFF = LD_OFF + 2 * LD_BYTES;
  // kv_full, qdo_full[3], qdo_empty[3], s_full, dp_full, p_ready[2], ds_ready[2], dq_full, dq_read,
  // dq_staged, dqb_empty, ld_ready[2], done
  static constexpr int NUM_BARS = 21;
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = MISC_OFF + 16 + 1024;  // + slack to align the base to 1024
  static constexpr uint32_t S_COL = 0, DP_COL = 128, DV_COL = 256, DK_COL = 320, DQ_COL = 384, K_COL = 448,
                            V_COL = 480;
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(BT, BT, false);
  static constexpr uint32_t IDESC_KV = idesc_bf16_f32(BT, D, true);
  static constexpr uint32_t IDESC_Q = idesc_bf16_f32(BT, D, true, true);
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

template <bool PACKED>
__global__ void __launch_bounds__(kBwdThreads)
    attn_bwd_tc64_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using C = Bwd64Cfg;
  constexpr int D = C::D, NST = C::NST;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_addr(smem_raw);
  const uint32_t pad = (1024u - (raw_s & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_s + pad;

  const uint32_t bar0 = sbase + C::BAR_OFF;
  const uint32_t bar_kv = bar0;
  auto bar_qdo = [&](int s) { return bar0 + 8u * (1 + s); };        // Q_i, dO_i of stage s landed
  auto bar_qdo_empty = [&](int s) { return bar0 + 8u * (4 + s); };  // the MMAs reading stage s complete
  const uint32_t bar_s = bar0 + 8u * 7;                             // S^T in TMEM
  const uint32_t bar_dp = bar0 + 8u * 8;                            // dP^T in TMEM
  auto bar_p = [&](int h) { return bar0 + 8u * (9 + h); };          // P^T of query half h in TMEM (4 warps)
  auto bar_ds = [&](int h) { return bar0 + 8u * (11 + h); };        // dS^T of half h in TMEM, dS staged
  const uint32_t bar_dq = bar0 + 8u * 13;                           // dQ in TMEM
  const uint32_t bar_dq_read = bar0 + 8u * 14;                      // dQ read out of TMEM (8 warps)
  const uint32_t bar_dq_staged = bar0 + 8u * 15;                    // dQ blocks staged (8 warps)
  const uint32_t bar_dqb_empty = bar0 + 8u * 16;                    // staged blocks read by their adds
  auto bar_ld = [&](int h) { return bar0 + 8u * (17 + h); };        // half h's (LSE, D) entries written
  const uint32_t bar_done = bar0 + 8u * 19;                         // every MMA of the CTA complete
  const uint32_t bar_kvt = bar0 + 8u * 20;                          // K, V copied into TMEM (8 warps)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  BwdGeom g;
  if (!bwd_geometry<PACKED>(p, g)) return;
  const int k0 = g.k0, Nq = g.Nq, Nk = g.Nk, qrow0 = g.qrow0, qplane0 = g.qplane0, n_it = g.n_it;
  const StepPos first_pos{0, g.i_begin};

  if (threadIdx.x == 0) {
    mbar_init(bar_kv, 1);
    for (int s = 0; s < NST; ++s) {
      mbar_init(bar_qdo(s), 1);
      mbar_init(bar_qdo_empty(s), 1);
    }
    mbar_init(bar_s, 1);
    mbar_init(bar_dp, 1);
    for (int h = 0; h < 2; ++h) {
      mbar_init(bar_p(h), kBwdRowWarps / 2);
      mbar_init(bar_ds(h), kBwdRowWarps / 2);
      mbar_init(bar_ld(h), kBwdRowWarps / 2);
    }
    mbar_init(bar_dq, 1);
    mbar_init(bar_dq_read, kBwdRowWarps);
    mbar_init(bar_dq_staged, kBwdRowWarps);
    mbar_init(bar_dqb_empty, 1);
    mbar_init(bar_done, 1);
    mbar_init(bar_kvt, kBwdRowWarps);
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
    tma_load_3d_elect(sbase + C::K_OFF, &tm_k, bar_kv, 0, g.krow0 + k0, g.kplane);
    tma_load_3d_elect(sbase + C::V_OFF, &tm_v, bar_kv, 0, g.krow0 + k0, g.kplane);
    int issued = 0, st = 0;
    uint32_t par = 0;  // step it uses stage st = it % NST for the (it / NST)-th time; par = that count & 1
    StepPos pos = first_pos;
    for (int it = 0; it < n_it; ++it, pos = pos.next(g)) {
      const int qp = qplane0 + pos.t, qy = qrow0 + pos.i * BT;
      // the stage's previous use (step it - NST) must be complete
      if (it >= NST && !(ok = wait_all(bar_qdo_empty(st), par ^ 1u, B_QDO_EMPTY))) break;
      mbar_arrive_expect_tx_elect(bar_qdo(st), 2 * C::TILE_BYTES);
      tma_load_3d_elect(sbase + C::Q_OFF + st * C::TILE_BYTES, &tm_q, bar_qdo(st), 0, qy, qp);
      tma_load_3d_elect(sbase + C::DO_OFF + st * C::TILE_BYTES, &tm_do, bar_qdo(st), 0, qy, qp);
      ++issued;
      if (++st == NST) {
        st = 0;
        par ^= 1u;
      }
    }
    // drain: every load issued must have landed before the CTA can exit
    for (int it = max(0, issued - NST); it < issued; ++it)
      mbar_wait(bar_qdo(it % NST), (uint32_t)(it / NST) & 1u, p.st, nullptr, (K_ATTN_BWD << 8) | B_DONE);
    mbar_wait(bar_kv, 0, p.st, nullptr, (K_ATTN_BWD << 8) | B_DONE);
  } else if (warp == kBwdMma) {
    // =================== MMA issue (whole warp, one elected lane) ===================
    // Descriptors are built once; a stage or K step only adds to the start-address field (shared
    // memory addresses >> 4 stay below 2^14, so the field never carries into the next one).
    const uint64_t k_nmaj = smem_desc_sw128(sbase + C::K_OFF, C::TILE_BYTES, 1024);      // B of dQ
    const uint64_t st_mmaj = smem_desc_sw128(sbase + C::ST_OFF, C::TILE_BYTES, 1024);    // A of dQ
    const uint64_t q_kmaj0 = smem_desc_sw128(sbase + C::Q_OFF, 16, 1024);
    const uint64_t do_kmaj0 = smem_desc_sw128(sbase + C::DO_OFF, 16, 1024);
    const uint64_t q_nmaj0 = smem_desc_sw128(sbase + C::Q_OFF, C::TILE_BYTES, 1024);
    const uint64_t do_nmaj0 = smem_desc_sw128(sbase + C::DO_OFF, C::TILE_BYTES, 1024);
    auto stage_off = [](int st) { return (uint64_t)((st * C::TILE_BYTES) >> 4); };
    auto kmaj = [&](int s0, int st, int kk) {  // K-major tile of stage st, K step kk (16 of the 64 dims)
      return (s0 == C::Q_OFF ? q_kmaj0 : do_kmaj0) + stage_off(st) + (uint64_t)((kk * 32) >> 4);
    };
    auto nmaj = [&](int s0, int st) { return (s0 == C::Q_OFF ? q_nmaj0 : do_nmaj0) + stage_off(st); };
    auto rows16_off = [](int kk) { return (uint64_t)((kk * 16 * 128) >> 4); };  // 16 rows of 128 bytes
    auto pcol = [](int kk) { return (uint32_t)(kk * 8 + (kk >= 4 ? 32 : 0)); };  // P^T / dS^T column
    // S^T (into S_COL, whose P^T the dV MMAs issued before have read) and dP^T (into DP_COL, whose
    // dS^T the dK MMAs issued before have read) of the step in stage st
    // A from TMEM: K (V) row k of the tile in lane k, dims 16 kk .. 16 kk + 15 in columns 8 kk .. + 7
    auto issue_s = [&](int st) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ts_elect(tmem_base + C::S_COL, tmem_base + C::K_COL + 8 * kk, kmaj(C::Q_OFF, st, kk), C::IDESC_S,
                     kk > 0 ? 1u : 0u);
      mma_commit_elect(bar_s);
    };
    auto issue_dp = [&](int st) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        mma_ts_elect(tmem_base + C::DP_COL, tmem_base + C::V_COL + 8 * kk, kmaj(C::DO_OFF, st, kk), C::IDESC_S,
                     kk > 0 ? 1u : 0u);
      mma_commit_elect(bar_dp);
    };
    bool ok = wait_all(bar_kv, 0, B_KV) && wait_all(bar_kvt, 0, B_KV);
    if (ok && n_it > 0 && (ok = wait_all(bar_qdo(0), 0, B_QDO))) {
      tc_fence_after_sync();
      issue_s(0);
      issue_dp(0);
    }
    int st = 0;
    uint32_t par = 0;
    for (int it = 0; ok && it < n_it; ++it) {
      const uint32_t ph = (uint32_t)it & 1u;
      const int st1 = st + 1 == NST ? 0 : st + 1;           // stage of step it + 1
      const uint32_t par1 = st1 == 0 ? par ^ 1u : par;
      const bool more = it + 1 < n_it;
      // dV += P^T dO_it once both halves of P^T are written
      if (!(ok = wait_all(bar_p(0), ph, B_DS) && wait_all(bar_p(1), ph, B_DS))) break;
      tc_fence_after_sync();
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int kk = 4 * h; kk < 4 * h + 4; ++kk)
          mma_ts_elect(tmem_base + C::DV_COL, tmem_base + C::S_COL + pcol(kk), nmaj(C::DO_OFF, st) + rows16_off(kk),
                       C::IDESC_KV, (it > 0 || kk > 0) ? 1u : 0u);
      }
      if (!ok) break;
      // the next step's S^T, so that the rows' next P pass need not wait for this step's dK / dQ
      if (more) {
        if (!(ok = wait_all(bar_qdo(st1), par1, B_QDO))) break;
        tc_fence_after_sync();
        issue_s(st1);
      }
      // dK += dS^T Q_it once both halves of dS^T are written
      if (!(ok = wait_all(bar_ds(0), ph, B_DS) && wait_all(bar_ds(1), ph, B_DS))) break;
      tc_fence_after_sync();
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int kk = 4 * h; kk < 4 * h + 4; ++kk)
          mma_ts_elect(tmem_base + C::DK_COL, tmem_base + C::DP_COL + pcol(kk), nmaj(C::Q_OFF, st) + rows16_off(kk),
                       C::IDESC_KV, (it > 0 || kk > 0) ? 1u : 0u);
      }
      if (!ok) break;
      // dQ_it = dS K_j into DQ_COL, once the rows have read dQ_{it-1} out of it
      if (it > 0 && !(ok = wait_all(bar_dq_read, ph ^ 1u, B_DQ_READ))) break;
      tc_fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < BT / 16; ++kk)
        mma_ss_elect(tmem_base + C::DQ_COL, st_mmaj + rows16_off(kk), k_nmaj + rows16_off(kk), C::IDESC_Q,
                     kk > 0 ? 1u : 0u);
      mma_commit_elect(bar_dq);
      mma_commit_elect(bar_qdo_empty(st));  // stage st free once this step's MMAs are complete
      if (more) issue_dp(st1);
      st = st1;
      par = par1;
    }
    // every MMA complete (for the dK / dV epilogue and before TMEM is freed)
    mma_commit_elect(bar_done);
    mbar_wait(bar_done, 0, p.st, nullptr, (K_ATTN_BWD << 8) | B_DONE);
  }
  else if (warp == kBwdReducer) {
    // ============ dQ reducer (whole warp, one lane issues): TMA reduce-adds of the blocks ============
    // Warp w's block of step it is added into rows q0 + 32 (w % 4) .. + 31 (clipped at Nq; skipped
    // when wholly past it) and columns 32 (w / 4) of the fp32 accumulator.
    bool ok = true;
    StepPos pos = first_pos;
    for (int it = 0; ok && it < n_it; ++it, pos = pos.next(g)) {
      const int q0 = pos.i * BT, qp = qplane0 + pos.t, qy = qrow0 + q0;
      if (!(ok = wait_all(bar_dq_staged, (uint32_t)it & 1u, B_DQ_STAGED))) break;
      if (lane == 0) {
        for (int w = 0; w < kBwdRowWarps; ++w) {
          if (q0 + (w & 3) * 32 >= Nq) continue;
          tma_reduce_add_3d(&tm_dq, sbase + C::DQB_OFF + w * 4096, (w >> 2) * 32, qy + (w & 3) * 32, qp);
        }
        bulk_commit_group();
        bulk_wait_read<0>();  // the buffer may be refilled once its blocks have been read
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_dqb_empty);
    }
    if (lane == 0) bulk_wait_all();  // every add performed before the CTA exits
    __syncwarp();
  } else {
    // =================== rows: warps 0-7, thread t = TMEM lane t % 128 ===================
    const int tt = threadIdx.x & (BT - 1);  // key row of the tile (the dQ tile: query row)
    const int half = warp >> 2;             // queries [64 half, 64 half + 64); dQ / dK / dV columns likewise
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tl = tmem_base + lane_base;
    const int key = k0 + tt;
    const bool key_ok = key < Nk;
    uint8_t* st_row = smem + C::ST_OFF + half * C::TILE_BYTES + tt * 128;  // key row in slab `half`
    // entries of the step with parity b: -LSE log2 e of its 128 queries, then -D scale
    auto nl4_of = [&](int b) { return reinterpret_cast<const float4*>(smem + C::LD_OFF + b * C::LD_BYTES); };
    auto nd4_of = [&](int b) { return reinterpret_cast<const float4*>(smem + C::LD_OFF + b * C::LD_BYTES + BT * 4); };
    // threads 0-63 of each half own the (LSE, D) entries of that half's queries
    const int ld_q = 64 * half + tt;
    // This warp's key rows of K (warps 0-3) or V (warps 4-7) into their TMEM columns, once: the
    // 128-byte row of the swizzled tile (16-byte chunk c of row r at chunk c ^ (r % 8)), as the bf16
    // pairs of the S^T / dP^T MMAs' A operand.
    {
      bool kv_ok = wait_all(bar_kv, 0, B_KV);
      if (kv_ok) {
        const uint8_t* trow = smem + (half ? C::V_OFF : C::K_OFF) + tt * 128;
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 u = *reinterpret_cast<const uint4*>(trow + ((c ^ (tt & 7)) * 16));
          w[4 * c] = u.x, w[4 * c + 1] = u.y, w[4 * c + 2] = u.z, w[4 * c + 3] = u.w;
        }
        tmem_st32(tl + (half ? C::V_COL : C::K_COL), w);
        tmem_st_wait();
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_kvt);
    }
    const uint64_t sl2x2 = f2_pack(p.scale_log2, p.scale_log2);
    const uint64_t sl2 = f2_pack(p.scale, p.scale);
    auto load_ld = [&](int step, StepPos sp, float& l, float& dd) {
      l = -INFINITY;
      dd = 0.f;
      const int q = sp.i * BT + ld_q;
      if (tt < 64 && step < n_it && q < Nq) {
        const int64_t row = g.lbase + (int64_t)q * g.lq + (int64_t)sp.t * g.lt;
        if (OA_DCHECK(p.st, row < p.lse_elems, (K_ATTN_BWD << 8) | (kSiteDebugBase + 1))) {
          l = p.lse[row];
          dd = p.dsum[row];
        }
      }
    };
    // -LSE log2 e and -D scale of a step's queries; a row past the end or with no visible key gets -inf,
    // so that exp2(s scale log2 e - inf) = 0 needs no test
    auto write_ld = [&](int b, float l, float dd) {
      if (tt < 64) {
        reinterpret_cast<float*>(smem + C::LD_OFF + b * C::LD_BYTES)[ld_q] = l == -INFINITY ? -INFINITY : -l * kLog2e;
        reinterpret_cast<float*>(smem + C::LD_OFF + b * C::LD_BYTES + BT * 4)[ld_q] = -dd * p.scale;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ld(half));
    };
    // dQ of step m out of TMEM (so that dQ of step m + 1 may follow), then staged as this warp's
    // 32 x 32 block (swizzled like the map) once the adds of step m - 1 have read the buffer
    auto drain_dq = [&](int m) {
      if (!wait_all(bar_dq, (uint32_t)m & 1u, B_DQ)) return false;
      tc_fence_after_sync();
      uint32_t r[32];
      tmem_ld32(tl + C::DQ_COL + half * 32, r);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_dq_read);
      if (m > 0 && !wait_all(bar_dqb_empty, (uint32_t)(m - 1) & 1u, B_DQ_STAGED)) return false;
      uint8_t* brow = smem + C::DQB_OFF + warp * 4096 + lane * 128;
#pragma unroll
      for (int q4 = 0; q4 < 8; ++q4)
        *reinterpret_cast<float4*>(brow + ((q4 ^ (lane & 7)) * 16)) =
            make_float4(__uint_as_float(r[4 * q4]), __uint_as_float(r[4 * q4 + 1]),
                        __uint_as_float(r[4 * q4 + 2]), __uint_as_float(r[4 * q4 + 3]));
      fence_proxy_async_smem();  // the blocks are read by the reducer warp's TMA (async proxy)
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_dq_staged);
      return true;
    };
    // the entries of step it go to buffer it % 2 during step it - 1, once this warp is past its dS
    // pass: every warp of the half has then read the entries of step it - 2 (it waited for all of them
    // to write the entries of step it - 1, which each does after its own dS pass of step it - 2);
    // their loads a step before that
    StepPos lpos = first_pos;
    float next_l, next_d;
    load_ld(0, lpos, next_l, next_d);
    write_ld(0, next_l, next_d);
    lpos = lpos.next(g);
    load_ld(1, lpos, next_l, next_d);
    bool ok = true;
    StepPos pos = first_pos;
    for (int it = 0; ok && it < n_it; ++it) {
      const int i = pos.i, q0 = i * BT;
      const uint32_t ph = (uint32_t)it & 1u;
      const bool full = (k0 + BT <= Nk) && (q0 + BT <= Nq) && (!p.causal || k0 + BT - 1 <= q0 + g.off);
      if (!(ok = wait_all(bar_s, ph, B_S))) break;
      if (!(ok = wait_all(bar_ld(half), ph, B_LD))) break;
      tc_fence_after_sync();
      // P^T of this warp's 64 queries over the first 32 of its S^T columns (read by it alone)
      const uint32_t sc = tl + C::S_COL + 64 * half;
      const uint32_t dc = tl + C::DP_COL + 64 * half;
      const float4* nl4 = nl4_of(it & 1);
      const float4* nd4 = nd4_of(it & 1);
      uint64_t pp[32];
      {
        uint32_t sr[64], pw[32];
        tmem_ld32x2(sc, sc + 32, sr);
        if (full)
          bwd_p<false>(sr, nl4 + 16 * half, sl2x2, key, q0 + 64 * half, true, false, pp, pw);
        else
          bwd_p<true>(sr, nl4 + 16 * half, sl2x2, key - g.off, q0 + 64 * half, key_ok, p.causal != 0, pp, pw);
        tmem_st32(sc, pw);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p(half));
      // the previous step's dQ (its MMA ran during this P pass); it also frees the dS buffer
      if (it > 0 && !(ok = drain_dq(it - 1))) break;
      if (!(ok = wait_all(bar_dp, ph, B_DP))) break;
      tc_fence_after_sync();
      {
        uint32_t dr[64], dw[32];
        tmem_ld32x2(dc, dc + 32, dr);
        bwd_ds(dr, nd4 + 16 * half, sl2, pp, dw);
        tmem_st32(dc, dw);
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8)
          *reinterpret_cast<uint4*>(st_row + ((q8 ^ (tt & 7)) * 16)) =
              make_uint4(dw[4 * q8], dw[4 * q8 + 1], dw[4 * q8 + 2], dw[4 * q8 + 3]);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      fence_proxy_async_smem();  // the staged dS is read by the tensor core (async proxy)
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ds(half));
      pos = pos.next(g);
      write_ld((it + 1) & 1, next_l, next_d);
      lpos = lpos.next(g);
      load_ld(it + 2, lpos, next_l, next_d);
    }
    if (ok && n_it > 0) ok = drain_dq(n_it - 1);
    if (ok && n_it > 0) ok = wait_all(bar_done, 0, B_DONE);
    if (ok) {
      tc_fence_after_sync();
      bwd_store_dkdv<D>(p, g, tl, C::DK_COL, C::DV_COL, half, key, key_ok, n_it > 0);
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

template <int D, bool PACKED>
cudaError_t launch_bwd_d(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                         const CUtensorMap& mdo, const CUtensorMap& mdq, const BwdParams& p, cudaStream_t s) {
  static bool attr_set[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const unsigned grid = (unsigned)p.nkt * (unsigned)p.BHkv;
  if constexpr (D == 64) {
    if (!attr_set[dev]) {
      e = cudaFuncSetAttribute(attn_bwd_tc64_kernel<PACKED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Bwd64Cfg::SMEM_BYTES);
      if (e != cudaSuccess) return e;
      attr_set[dev] = true;
    }
    attn_bwd_tc64_kernel<PACKED><<<grid, kBwdThreads, Bwd64Cfg::SMEM_BYTES, s>>>(mq, mk, mv, mdo, mdq, p);
  } else {
    if (!attr_set[dev]) {
      e = cudaFuncSetAttribute(attn_bwd_tc_kernel<D, PACKED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               BwdCfg<D>::SMEM_BYTES);
      if (e != cudaSuccess) return e;
      attr_set[dev] = true;
    }
    attn_bwd_tc_kernel<D, PACKED><<<grid, kBwdThreads, BwdCfg<D>::SMEM_BYTES, s>>>(mq, mk, mv, mdo, mdq, p);
  }
  return cudaGetLastError();
}

}  // namespace

size_t attn_bwd_workspace_floats(int B, int H, int Nq, int d) { return (size_t)B * H * Nq * ((size_t)d + 1); }

cudaError_t launch_attn_bwd(const BwdArgs& a, float* workspace, const DevStatus& st, cudaStream_t s,
                            const char** why) {
  // dense: [B, H, N, d] (planes of N rows); packed: [tokens, H, d] (rows of H d elements, heads as
  // planes), B = 1 and Nq, Nk the token counts
  const bool packed = a.cu_q != nullptr;
  const int d = a.d, BH = a.B * a.H, BHkv = a.B * a.Hkv;
  const int64_t eb = 2 * (int64_t)d;  // bytes per row of one head
  const int64_t rows = (int64_t)BH * a.Nq;
  float* dq_acc = workspace;
  float* dsum = workspace + rows * d;
  const int64_t q_row = packed ? eb * a.H : eb, q_plane = packed ? eb : eb * a.Nq;
  const int64_t k_row = packed ? eb * a.Hkv : eb, k_plane = packed ? eb : eb * a.Nk;
  CUtensorMap mq, mk, mv, mdo, mdq;
  if (!make_tile_map(&mq, a.q, d, a.Nq, q_row, BH, q_plane) ||
      !make_tile_map(&mk, a.k, d, a.Nk, k_row, BHkv, k_plane) ||
      !make_tile_map(&mv, a.v, d, a.Nk, k_row, BHkv, k_plane) ||
      !make_tile_map(&mdo, a.dout, d, a.Nq, q_row, BH, q_plane) ||
      !make_f32_tile_map(&mdq, dq_acc, d, a.Nq, 2 * q_row, BH, 2 * q_plane, 32)) {
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
  p.nkt = ((packed ? a.max_seqlen_k : a.Nk) + BT - 1) / BT;
  p.nqt = (a.Nq + BT - 1) / BT;
  p.BHkv = packed ? a.num_seqs * a.Hkv : BHkv;
  p.group = a.H / a.Hkv;
  p.H = a.H;
  p.Hkv = a.Hkv;
  p.cu_q = a.cu_q;
  p.cu_k = a.cu_k;
  p.total_q = a.Nq;
  p.total_k = a.Nk;
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.lse_elems = rows;
  p.dk_elems = (int64_t)(packed ? 1 : a.B) * a.Hkv * a.Nk * d;
  p.st = st;
  if (p.nkt < 1) p.nkt = 1;
  if (packed)
    e = d == 128 ? launch_bwd_d<128, true>(mq, mk, mv, mdo, mdq, p, s)
                 : launch_bwd_d<64, true>(mq, mk, mv, mdo, mdq, p, s);
  else
    e = d == 128 ? launch_bwd_d<128, false>(mq, mk, mv, mdo, mdq, p, s)
                 : launch_bwd_d<64, false>(mq, mk, mv, mdo, mdq, p, s);
  if (e != cudaSuccess) return e;
  const int64_t n = rows * d;
  bwd_post_kernel<<<(unsigned)((n / 4 + 255) / 256), 256, 0, s>>>(dq_acc, static_cast<__nv_bfloat16*>(a.dq), n);
  return cudaGetLastError();
}

}  // namespace oa
