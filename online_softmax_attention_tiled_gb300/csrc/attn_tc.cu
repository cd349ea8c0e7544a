// attn_tc.cu -- fused attention forward on the 5th-generation tensor cores
// (tcgen05, tensor memory) for bf16 inputs, fp32 accumulation, d = 64 / 128.
//
// Method: the attention promotion of the online softmax (roadmap page s.5;
// research-hub page "Key math"): per query row a running max m, running
// denominator l and unnormalised output o; for each key/value tile
//   m_new = max(m_old, rowmax(S)), alpha = exp(m_old - m_new),
//   P = exp(S - m_new), l = alpha l + rowsum(P), o = alpha o + P V,
// and o / l, LSE = m + ln l once at the end.  The loop order is Q-outer
// (interview lesson Step 3): one CTA owns 256 query rows of one (b, h) and
// streams the key/value tiles past them; the score tile never leaves the
// chip.  Causal: the Nq queries are the last Nq positions of the Nk keys'
// sequence (new tokens after a KV cache), so query i sees keys
// j <= i + (Nk - Nq) -- per sequence for packed sequences.  Key tiles past
// a query tile's last visible key are never loaded or computed; only the
// tiles the diagonal crosses and the ragged key tail are masked (Step 4).
//
// Persistent: one CTA per SM, each working through items (2 x 128 query rows of one
// (b, h)) numbered heaviest first and dealt out in rounds of one per CTA, alternating
// direction between rounds.  Causal launches whose K/V exceeds L2 sweep bands of heads in
// phases (each phase dealt this way, odd phases in mirrored CTA order; the host picks the count
// for the dense layout, the kernel from the sequence lengths for packed sequences), and odd
// rounds read the key tiles top down, so K/V is read from DRAM about once.  Q and O, read and written
// once, carry an evict-first L2 policy.  Barriers, TMEM and descriptors are set up once; ring
// loads and barrier phases run on across items, so the next item's Q, K and V are loaded and
// its first score tiles computed while the current item finishes.
//
// GB300 mapping (352 threads; 320 at d = 128 with two query tiles):
//   warps 0-3   softmax for query tile 0 (rows q0 .. q0+127): thread t owns
//               row t, i.e. TMEM lane t, so row max / sum are thread-local
//   warps 4-7   softmax for query tile 1 (rows q0+128 .. q0+255)
//   warp 8      TMA producer: Q per item, then K and V tiles into one 4-slot
//               (d=128) / 10-slot (d=64) shared-memory ring in load order
//               K0,V0,K1,V1,... (128-byte swizzle), mbarrier complete_tx
//   warps 9, 10 MMA issue for query tile 0 / 1 (whole warp, one elected lane):
//               S_i = Q_i K^T (SMEM x SMEM -> TMEM) and O_i += P_i V (P from
//               TMEM, V from SMEM -> TMEM); warp 9 owns the TMEM allocation.
//               One warp issues an N <= 128 MMA in about 70 (A from shared
//               memory) to 90 (A from TMEM) cycles, a little longer than the
//               64 the tensor core takes for an N = 128 one and two to three
//               times the 32 of an N = 64 one, so each tile has its own issuer
//               -- except at d = 128 with two query tiles, where warp 9 alone
//               issues both tiles' MMAs (see Cfg::mma_warps)
// TMEM (512 columns x 128 lanes, fp32): S_0 [0,128), S_1 [128,256),
// O_0 [256, 256+d), O_1 [256+d, 256+2d).
//   d = 128: P_i (bf16, two per column) is written over the first 64 columns
//   of S_i, so S_i(j+1) can only follow the PV MMA that reads P_i(j).  Warp 9
//   issues PV_0(j), S_0(j+1), PV_1(j), S_1(j+1) (the split-slot instances: each
//   slot's warp its own), and each softmax group works while the tensor core
//   runs the other group's MMAs.  PV_i(j) goes in two halves: keys 0-63 once
//   the group has handed over the first half of P_i (p_half), keys 64-127 once
//   all of P_i is written (p_full).
//   d = 64: P_i gets its own columns [384 + 64 i, +64), so the group frees
//   S_i as soon as it has read it and S_i(j+1) is computed during the
//   softmax of S_i(j): the order is S_i(j+1), PV_i(j); before writing P_i(j)
//   a group waits for PV_i(j-1).
//   SPLIT instances (dense, at most 128 query rows: decode, multi-token decode):
//   an item would fill only query tile 0, so both tiles hold the same rows
//   and take alternate key tiles (tile 0 the even, tile 1 the odd ones) with
//   their own (m, l, O); at the end group 1 hands (m, l) to group 0 through
//   Q tile 1's buffer, which this mode never loads, and group 0 merges the
//   two partial results (the same (m, l) merge as split-KV) and writes O.
//
// Every mbarrier wait is bounded (oa_common.cuh); a wait that expires sets
// the CTA abort flag, every role falls through to the teardown, in-flight
// TMA loads and MMAs are drained (bounded), and TMEM is always freed.
#include "oa_internal.h"

#include <algorithm>
#include <vector>

namespace oa {
namespace {

constexpr int BM = 128;  // rows per query tile (= TMEM lanes)
// Keys per key/value tile at d = 128.  128: P_i is written over S_i, and each tile's softmax, PV and
// next S follow one another.  64 would fit S tiles (64 columns each), O tiles (128 each) and separate
// P columns (32 each) in the 512 TMEM columns and run the pipeline of d = 64 (S_i(j+1) computed
// while the softmax of S_i(j) runs from registers); it measured 4 % slower at causal N = 8192: a
// group's softmax of a 64-key tile costs about 80 % of a 128-key one (fixed per-tile latencies), and
// the S MMAs at N = 64 take more MMA issue slots from the softmax warps that share their SMSPs.
constexpr int kD128KeysPerTile = 128;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp0 = 9;  // MMA issuer of query tile 0; warp 10 issues for tile 1
constexpr uint32_t kTmemCols = 512;
// A row's running max is only moved (and O, l rescaled) when a tile raises it
// by more than this many log2 units, i.e. a factor 2^8.
constexpr float kRescaleLog2 = 8.f;
// P over S: pairs of P computed after the first half of P is stored and before that half is handed
// to the MMA warp (causal N = 8192, d = 128: 0 or 8 pairs 1540 TFLOP/s, 16 pairs 1544-1549)
constexpr int kPHandoffLag = 16;

template <int D>
struct Cfg {
  static constexpr int BN = (D == 128) ? kD128KeysPerTile : 128;  // keys per key/value tile
  static constexpr int SLABS = D / 64;               // 128-byte swizzle atoms along d
  static constexpr int Q_SLAB = BM * 128;            // 128 rows x 128 bytes
  static constexpr int KV_SLAB = BN * 128;           // BN rows x 128 bytes
  static constexpr int Q_TILE = SLABS * Q_SLAB;
  static constexpr int KV_TILE = SLABS * KV_SLAB;
  // One ring of key/value tiles, filled in the order the MMAs consume them:
  // K_0, V_0, K_1, V_1, ... (load t = 2j for K_j, 2j + 1 for V_j, slot t % SLOTS).
  static constexpr int SLOTS = (KV_TILE <= 16384) ? 10 : 4;
  // When S_0, S_1 (BN columns each), O_0, O_1 (D each) and P_0, P_1 (BN / 2 each, bf16 pairs)
  // fit the 512 columns, P_i gets columns of its own, so S_i(j+1) can be computed while the
  // softmax of S_i(j) runs (the group frees S_i as soon as it has read it).  Else P_i is
  // written over S_i.
  static constexpr bool SEP_P = (3 * BN + 2 * D <= 512);
  // MMA issuing warps: one per query tile, except with P_i over S_i in the two-tile (non-SPLIT)
  // instances, where one warp issues both tiles' MMAs: a tile's PV_i(j), S_i(j+1) then run back to
  // back instead of interleaved with the other tile's, which keeps each tile's critical loop
  // (softmax -> PV_i -> S_i -> softmax) short (measured 12 % faster than two issuers at causal
  // N = 8192, d = 128).
  template <bool SPLIT>
  static constexpr int mma_warps() { return (!SEP_P && !SPLIT) ? 1 : 2; }
  template <bool SPLIT>
  static constexpr int threads() { return 32 * (9 + mma_warps<SPLIT>()); }  // 8 softmax warps, producer
  static constexpr int Q_OFF = 0;
  static constexpr int RING_OFF = Q_OFF + 2 * Q_TILE;
  static constexpr int BAR_OFF = RING_OFF + SLOTS * KV_TILE;
  // With P_i over S_i the group hands P_i over in two halves: the PV MMAs of the first half of the
  // keys are issued while the group still computes the second half.
  static constexpr bool HALF_P = !SEP_P;
  // q_full, full[SLOTS], empty[SLOTS], s_full[2], p_full[2], o_done[2], drain, s_free[2], q_empty,
  // p_half[2]
  static constexpr int NUM_BARS = 1 + 2 * SLOTS + 6 + 1 + 2 + 1 + 2;
  static constexpr int MISC_OFF = BAR_OFF + NUM_BARS * 8;
  // MISC: TMEM address (4 bytes), abort flag (4), at 16 a PackedDeal (12)
  static constexpr int SMEM_BYTES = MISC_OFF + 32 + 1024;  // + slack to align the base to 1024
  __host__ __device__ static constexpr uint32_t s_col(int i) { return (uint32_t)(i * BN); }
  __host__ __device__ static constexpr uint32_t o_col(int i) { return (uint32_t)(2 * BN + i * D); }
  // first TMEM column of P_i (bf16 pairs, BN / 2 columns)
  __host__ __device__ static constexpr uint32_t p_col(int i) {
    return SEP_P ? (uint32_t)(2 * BN + 2 * D + i * (BN / 2)) : s_col(i);
  }
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, false);  // Q K^T, both K-major
  static constexpr uint32_t IDESC_O = idesc_bf16_f32(BM, D, true);    // P V, V is MN-major
  static_assert(BN == 64 || BN == 128, "key tile");
  static_assert(SEP_P ? 3 * BN + 2 * D <= (int)kTmemCols : 2 * BN + 2 * D <= (int)kTmemCols, "TMEM columns");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

struct TcParams {
  __nv_bfloat16* o;
  float* lse;
  const int32_t* kv_len;  // dense layout: keys per batch entry, or NULL
  // Packed sequences (NULL: the dense [B, H, N, d] layout): sequence s has query tokens
  // [cu_q[s], cu_q[s+1]) of q [Tq, H, d] and key tokens [cu_k[s], cu_k[s+1]) of k/v [Tk, H_kv, d].
  const int32_t* cu_q;
  const int32_t* cu_k;
  int Tq, Tk;
  int H, Nq, Nk, num_qblocks, BH;  // packed: Nq = longest query sequence, BH = sequences x H
  int off;               // dense causal: query i sees keys j <= i + off (Nk - Nq); causality is the MODE
  int qmod;              // > 0: a row's causal position is its index modulo qmod (grouped decode rows)
  int group;             // query heads per key/value head (H / H_kv)
  // Heaviest-first items are dealt in n_groups phases, each over the heads of a band of
  // key/value planes (group_items items, group_rounds rounds of the grid); 1 phase otherwise
  int n_groups, group_items, group_rounds;
  // The key-tile order of a causal item follows the round it has in the dealing of the whole call
  // (dir_hs heads a phase, dir_G CTAs), in which this launch's head plane 0 is plane dir_sh0
  int dir_hs, dir_G, dir_sh0;
  int dir_alt;  // 0: every item reads its key tiles bottom up (a call dealt plane by plane)
  int call_bh, call_sh0;  // the whole call's planes and this launch's first (host side, see TcArgs)
  int plane_major;        // kCausalOff, dense, one phase: items numbered plane by plane (see item_at)
  int decide_phases;      // packed causal: the kernel picks the phase count from the sequence lengths
  int64_t o_rs;          // O row stride (elements): d dense, H d packed
  int64_t o_elems, lse_elems;  // extents of o and lse (the debug build's store checks)
  int l_rs;              // LSE row stride: 1 dense, H packed
  int o_v8;  // o is 32-byte aligned: rows are written with 32-byte stores
  float scale_log2;
  DevStatus st;
};

enum WaitSite : unsigned {
  W_Q = 1, W_KFULL, W_KEMPTY, W_VFULL, W_VEMPTY, W_SFULL, W_PFULL, W_ODONE, W_DRAIN, W_SFREE, W_QEMPTY
};

// Masking mode, a template parameter of the kernel (each mode compiles to its own instance):
//   kNonCausal  every key up to the sequence's length; items are numbered head-major, so the items
//               of one key/value plane run together and share its K/V in L2
//   kCausal     square causal (Nq == Nk, key offset 0), heaviest query blocks first
//   kCausalOff  causal with a key offset (Nq != Nk, or packed sequences, each with its own)
// A runtime offset in the mask measured 3 % slower on the square causal case, and a runtime
// choice of the item order 1 % slower, hence three instances.
enum Mode : int { kNonCausal = 0, kCausal = 1, kCausalOff = 2 };

// One work item: 2 x 128 query rows of one (sequence, head).
struct Item {
  int zq, zkv;      // tensor-map head plane of Q/O and of K/V
  int yq, ykv;      // tensor-map row of the sequence's first query / key
  int q0;           // first query row of the item within its sequence
  int nq, kvl;      // query rows and keys of the sequence
  int off;          // causal: query i sees keys j <= i + off (keys minus queries of the sequence)
  int n_kv[2], n_all;
  int nrev;         // key tiles read in descending order: load L < nrev holds key tile nrev - 1 - L
  int64_t ob, lb;   // offsets of the sequence's row 0 (this head) in O (elements) and in LSE
};

// Causal launches deal their items in phases over bands of heads (see item_of); the others in
// one.  Dense: the host picks the phase count; packed: the kernel does, from the sequence lengths
// (PackedDeal).
template <bool PACKED, bool SPLIT, int MODE>
constexpr bool phased() { return !SPLIT && MODE != kNonCausal; }

// The dealing of a packed causal launch, decided by every CTA at its start (see the kernel).
struct PackedDeal {
  int phases, items, rounds;  // phase count, items per phase, rounds of the grid per phase
};

// Items are numbered heaviest first (causal, and packed sequences: the last query blocks) within
// each phase: item idx = f * group_items + r of phase f covers query block num_qblocks - 1 - r / hs
// of (sequence, head) f * hs + r % hs, hs = BH / n_groups heads per phase (all of them with one
// phase).
// Dense non-causal items weigh alike and are numbered head-major: query block idx % num_qblocks
// of head plane idx / num_qblocks.  Query head h reads key/value head h / group.  SPLIT (at most
// 128 query rows): both query-tile slots hold the same rows, slot 0 takes the even key tiles and
// slot 1 the odd ones.
template <int D, bool PACKED, bool SPLIT, int MODE>
__device__ __forceinline__ Item item_at(const TcParams& p, int idx, const PackedDeal* pd) {
  constexpr int BN = Cfg<D>::BN;
  Item it;
  constexpr bool kHeadMajor = !PACKED && MODE == kNonCausal;
  constexpr bool kPhased = phased<PACKED, SPLIT, MODE>();
  const int n_groups = (PACKED && kPhased) ? pd->phases : p.n_groups;
  const int group_items = (PACKED && kPhased) ? pd->items : p.group_items;
  const int phase = kPhased ? idx / group_items : 0;
  const int r = idx - phase * group_items, hs = kPhased ? p.BH / n_groups : p.BH;
  // a causal launch with a key offset whose items weigh nearly alike (a chunk of queries after a
  // long cache) numbers them plane by plane, heaviest first within a plane: the items running at
  // the same time then share few K/V planes
  const bool by_plane = MODE == kCausalOff && kPhased && p.plane_major;
  const int qb = kHeadMajor ? idx % p.num_qblocks
                            : p.num_qblocks - 1 - (by_plane ? r % p.num_qblocks : r / hs);
  const int sh = kHeadMajor ? idx / p.num_qblocks : by_plane ? r / p.num_qblocks : phase * hs + r % hs;
  const int sq = sh / p.H, h = sh % p.H, hk = h / p.group;
  const int Hkv = p.H / p.group;
  it.q0 = qb * 2 * BM;
  if constexpr (PACKED) {
    // lengths are clamped to the tensors, so a bad offset can only drop rows, never
    // address outside q, k, v, o or lse
    const int q_beg = min(max(p.cu_q[sq], 0), p.Tq), q_end = min(max(p.cu_q[sq + 1], q_beg), p.Tq);
    const int k_beg = min(max(p.cu_k[sq], 0), p.Tk), k_end = min(max(p.cu_k[sq + 1], k_beg), p.Tk);
    it.nq = q_end - q_beg;
    it.kvl = k_end - k_beg;
    it.off = it.kvl - it.nq;
    if (it.nq > p.Nq) {  // longer than the declared maximum: its tail has no items
      if (qb == 0 && h == 0) record_failure(p.st, kSiteBadSeqlen);
      it.nq = p.Nq;
    }
    it.zq = h;
    it.zkv = hk;
    it.yq = q_beg;
    it.ykv = k_beg;
    it.ob = ((int64_t)q_beg * p.H + h) * D;
    it.lb = (int64_t)q_beg * p.H + h;
  } else {
    it.nq = p.Nq;
    it.kvl = p.Nk;
    it.off = MODE == kCausalOff ? p.off : 0;  // from the shapes (Nk - Nq); kv_len only hides the tail
    if (p.kv_len != nullptr) it.kvl = min(max(p.kv_len[sq], 0), p.Nk);
    it.zq = sh;
    it.zkv = sq * Hkv + hk;
    it.yq = 0;
    it.ykv = 0;
    it.ob = (int64_t)sh * p.Nq * D;
    it.lb = (int64_t)sh * p.Nq;
  }
  const int nk_tiles = (it.kvl + BN - 1) / BN;
  // Key tiles a query tile reads: causal, up to the tile holding key r_last + off, r_last being the
  // tile's last row (past nq its rows are computed and dropped, so the count for Nq == Nk is that of
  // a square diagonal); none when that key is negative.  Else every tile.
  auto tiles_to = [&](int r_last) {
    return MODE == kNonCausal ? nk_tiles : max(0, min(nk_tiles, (r_last + it.off + BN) / BN));
  };
  if constexpr (SPLIT) {
    const int nt = it.q0 < it.nq ? tiles_to(it.q0 + BM - 1) : 0;
    it.n_kv[0] = (nt + 1) / 2;
    it.n_kv[1] = nt / 2;
  } else {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int r0 = it.q0 + i * BM;
      it.n_kv[i] = r0 < it.nq ? tiles_to(r0 + BM - 1) : 0;  // none past the end
    }
  }
  it.n_all = max(it.n_kv[0], it.n_kv[1]);
  // Causal items of odd rounds read the key tiles that both query tiles share from the top down
  // (the longer tile's extra tiles still come last, so both tiles start at the item's first load
  // and the shorter one stops early).  Every round starts a new item on every CTA; read from the
  // bottom, a round would begin on the key tiles the previous round read first, which L2 has
  // evicted by then when the phase's K/V does not fit, and re-read them from DRAM.  Starting
  // from the top it begins on the tiles the previous round read last.  The online softmax does
  // not depend on the order of the key tiles.
  it.nrev = 0;
  if constexpr (!SPLIT && MODE != kNonCausal) {
    // an odd round of the item's phase in the dealing of the whole call: this launch's own,
    // unless it is a piece of a dense call cut into pieces (dir_*); a packed launch is always a
    // whole call
    const int dir_hs = PACKED ? hs : p.dir_hs, dir_G = PACKED ? (int)gridDim.x : p.dir_G;
    const int dir_sh0 = PACKED ? 0 : p.dir_sh0;
    if ((PACKED || p.dir_alt) && ((((p.num_qblocks - 1 - qb) * dir_hs + (dir_sh0 + sh) % dir_hs)) / dir_G) & 1) {
      const int a = it.n_kv[0], b = it.n_kv[1];
      it.nrev = (a > 0 && b > 0) ? min(a, b) : it.n_all;
    }
  }
  return it;
}

// The key tile held by the item's L-th K/V load.
__device__ __forceinline__ int key_tile(int L, int nrev) { return L < nrev ? nrev - 1 - L : L; }

// Key tiles an item loads (K_0, V_0, K_1, V_1, ...): each once, shared by both slots, or (SPLIT)
// split between them.
template <bool SPLIT>
__device__ __forceinline__ int n_loads_of(const Item& it) { return SPLIT ? it.n_kv[0] + it.n_kv[1] : it.n_all; }

// The k-th item of this CTA.  Phase f = k / group_rounds runs after phase f - 1 on every CTA;
// round k' = k % group_rounds of a phase takes its items [k' G, k' G + G), in CTA order on even
// rounds and in reverse on odd ones, so the heavy and light ends of the phase's list pair up
// across rounds; odd phases deal in mirrored CTA order, so that the last, partial rounds of two
// consecutive phases fall on CTAs at opposite ends of the grid.  Negative past the end of a
// phase.  (One phase: item k G + c or k G + G - 1 - c of the whole list.)
template <bool PHASED>
__device__ __forceinline__ int item_of(int k, int group_items, int group_rounds) {
  const int G = (int)gridDim.x;
  const int f = PHASED ? k / group_rounds : 0, kr = k - f * group_rounds;
  const int c = (f & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x;
  const int r = kr * G + ((kr & 1) ? (G - 1 - c) : c);
  return r < group_items ? f * group_items + r : -1;
}

// Key tiles an item of query block qb of a packed sequence with nq_raw queries and kvl keys
// loads (n_all of item_at; nq_raw above the declared maximum Nq is cut to it there).
template <int D>
__device__ __forceinline__ int packed_item_tiles(int nq_raw, int kvl, int qb, int Nq) {
  constexpr int BN = Cfg<D>::BN;
  const int off = kvl - nq_raw, nq = min(nq_raw, Nq), nk_tiles = (kvl + BN - 1) / BN;
  int n = 0;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r0 = qb * 2 * BM + i * BM;
    if (r0 < nq) n = max(n, max(0, min(nk_tiles, (r0 + BM - 1 + off + BN) / BN)));
  }
  return n;
}

// x / y for 0 <= x < 2^22 and 1 <= y, by a float reciprocal and one correction each way.
__device__ __forceinline__ int small_div(int x, int y, float inv_y) {
  int q = __float2int_rz(__int2float_rn(x) * inv_y);
  if (q * y > x) --q;
  if ((q + 1) * y <= x) ++q;
  return q;
}

// No minimum-blocks hint: one CTA per SM follows from the shared memory and TMEM it takes,
// and the hint made ptxas spill more on this kernel.  PACKED: token-major packed sequences
// (a separate instance, so the dense layout pays nothing for them).  MODE: see Mode.
template <int D, bool PACKED, bool SPLIT, int MODE>
__global__ void __launch_bounds__(Cfg<D>::template threads<SPLIT>())
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const TcParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_addr(smem_raw);
  const uint32_t pad = (1024u - (raw_s & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_s + pad;

  const uint32_t bar0 = sbase + C::BAR_OFF;
  const uint32_t bar_q = bar0;
  auto bar_full = [&](int t) { return bar0 + 8u * (1 + t % C::SLOTS); };             // ring load t landed
  auto bar_empty = [&](int t) { return bar0 + 8u * (1 + C::SLOTS + t % C::SLOTS); };  // slot of load t free
  auto ring_phase = [&](int t) { return (uint32_t)(t / C::SLOTS) & 1u; };
  auto ring_addr = [&](int t) { return sbase + C::RING_OFF + (uint32_t)((t % C::SLOTS) * C::KV_TILE); };
  auto bar_sfull = [&](int i) { return bar0 + 8u * (1 + 2 * C::SLOTS + i); };
  auto bar_pfull = [&](int i) { return bar0 + 8u * (3 + 2 * C::SLOTS + i); };
  auto bar_odone = [&](int i) { return bar0 + 8u * (5 + 2 * C::SLOTS + i); };
  const uint32_t bar_drain = bar0 + 8u * (7 + 2 * C::SLOTS);
  auto bar_sfree = [&](int i) { return bar0 + 8u * (8 + 2 * C::SLOTS + i); };  // S_i read by its group
  const uint32_t bar_qempty = bar0 + 8u * (10 + 2 * C::SLOTS);               // Q read by the last S MMAs
  auto bar_phalf = [&](int i) { return bar0 + 8u * (11 + 2 * C::SLOTS + i); };  // first half of P_i written
  static_assert(!SPLIT || !PACKED, "the split mode serves the dense layout");
  // SPLIT: Q tile 1's buffer (never loaded) holds group 1's (m, l) per row and two barriers:
  // xch (group 1's O_1, m, l ready; 4 warps) and xdone (group 0 has read them; 4 warps)
  float2* xch_ml = reinterpret_cast<float2*>(smem + C::Q_OFF + C::Q_TILE);
  const uint32_t bar_xch = sbase + C::Q_OFF + C::Q_TILE + BM * 8;
  const uint32_t bar_xdone = bar_xch + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr bool kPhased = phased<PACKED, SPLIT, MODE>();
  PackedDeal* pdeal = reinterpret_cast<PackedDeal*>(smem + C::MISC_OFF + 16);
  constexpr int kIssuers = C::template mma_warps<SPLIT>();
  constexpr bool kOneIssuer = kIssuers == 1;

  // ---- set-up: barriers, TMEM (once; the CTA then works through its items) ----
  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int t = 0; t < C::SLOTS; ++t) {
      mbar_init(bar_full(t), 1);
      mbar_init(bar_empty(t), kIssuers);  // released by every MMA warp
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_sfull(i), 1);
      mbar_init(bar_pfull(i), 4);  // one arrival per softmax warp
      mbar_init(bar_odone(i), 1);
      mbar_init(bar_sfree(i), 4);  // one arrival per softmax warp
      mbar_init(bar_phalf(i), 4);  // one arrival per softmax warp
    }
    mbar_init(bar_drain, kIssuers);
    mbar_init(bar_qempty, kIssuers);
    if constexpr (SPLIT) {
      mbar_init(bar_xch, 4);
      mbar_init(bar_xdone, 4);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp0) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  if constexpr (PACKED && kPhased) {
    // ---- the dealing of a packed causal launch, decided alike by every CTA ----
    // When the K/V does not fit in L2 (decide_phases), every CTA simulates the dealing with 1, 4
    // and 16 phases over bands of (sequence, head) planes -- weights: the key tiles an item loads
    // plus two -- and takes the largest count that leaves the busiest CTA at most 0.5 % busier
    // than one phase does (simulated over random batches, the phases balanced 1-2 % better on
    // average and read K/V from DRAM 3-4x less; 16 packed sequences of 1894-8091 tokens, H32
    // H_kv 8: 1.6 % faster over 3 s under the power cap, from a higher clock with 2.8x less DRAM
    // traffic, at 3 % more SM cycles).  The weight table and loads live in the K/V ring, which no
    // TMA load has touched yet.  Any count dividing the planes is a valid dealing; the choice only
    // affects speed.
    constexpr int kTable = 16384;  // (sequence, query block) weights at most
    constexpr int kCands[3] = {1, 4, 16};
    const int G = (int)gridDim.x, NQB = p.num_qblocks, BH = p.BH, S = p.BH / p.H;
    // scratch in the ring: lengths (2 S ints), weights (S NQB ints), loads (3 G long longs)
    const long long w_off = (8ll * S + 15) / 16 * 16, l_off = (w_off + 4ll * S * NQB + 15) / 16 * 16;
    const bool decide = p.decide_phases != 0 && (long long)S * NQB <= kTable &&
                        (long long)BH * NQB <= (1ll << 22) && l_off + 24ll * G <= (long long)C::SLOTS * C::KV_TILE;
    if (decide) {
      int* lens = reinterpret_cast<int*>(smem + C::RING_OFF);  // queries, keys of each sequence
      int* W = reinterpret_cast<int*>(smem + C::RING_OFF + w_off);
      long long* load = reinterpret_cast<long long*>(smem + C::RING_OFF + l_off);
      for (int sq = threadIdx.x; sq < S; sq += blockDim.x) {
        // lengths clamped as item_at clamps them
        const int q_beg = min(max(p.cu_q[sq], 0), p.Tq), q_end = min(max(p.cu_q[sq + 1], q_beg), p.Tq);
        const int k_beg = min(max(p.cu_k[sq], 0), p.Tk), k_end = min(max(p.cu_k[sq + 1], k_beg), p.Tk);
        lens[2 * sq] = q_end - q_beg;
        lens[2 * sq + 1] = k_end - k_beg;
      }
      __syncthreads();
      for (int e = threadIdx.x; e < S * NQB; e += blockDim.x) {
        const int sq = e / NQB, qb = e - sq * NQB;
        const int n = packed_item_tiles<D>(lens[2 * sq], lens[2 * sq + 1], qb, p.Nq);
        W[e] = n > 0 ? n + 2 : 0;
      }
      __syncthreads();
      const float inv_h = 1.f / (float)p.H;
      for (int task = threadIdx.x; task < 3 * G; task += blockDim.x) {
        const int ci = task / G, b = task - ci * G, ng = kCands[ci];
        long long sum = -1;  // -1: the count does not divide the planes, or a phase is under 2 rounds
        if (BH % ng == 0 && (BH / ng) % p.group == 0 && (ng == 1 || (long long)(BH / ng) * NQB >= 2ll * G)) {
          const int hs = BH / ng, gi = hs * NQB, gr = (gi + G - 1) / G;
          const float inv_hs = 1.f / (float)hs;
          sum = 0;
          for (int f = 0; f < ng; ++f) {
            const int c = (f & 1) ? G - 1 - b : b;
#pragma unroll 4
            for (int kr = 0; kr < gr; ++kr) {
              const int r = kr * G + ((kr & 1) ? (G - 1 - c) : c);
              if (r >= gi) continue;
              const int lvl = small_div(r, hs, inv_hs), sh = f * hs + (r - lvl * hs);
              sum += W[small_div(sh, p.H, inv_h) * NQB + (NQB - 1 - lvl)];
            }
          }
        }
        load[ci * G + b] = sum;
      }
      __syncthreads();
      if (warp == 0) {  // the busiest CTA of each count (-1: the count is not allowed)
        long long mx[3];
#pragma unroll
        for (int ci = 0; ci < 3; ++ci) {
          long long m = 0;
          for (int b = lane; b < G; b += 32) m = (load[ci * G + b] < 0 || m < 0) ? -1 : max(m, load[ci * G + b]);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const long long x = __shfl_xor_sync(0xffffffffu, m, o);
            m = (x < 0 || m < 0) ? -1 : max(m, x);
          }
          mx[ci] = m;
        }
        if (lane == 0) {
          int best = 1;
#pragma unroll
          for (int ci = 1; ci < 3; ++ci)
            if (mx[ci] >= 0 && mx[ci] * 1000 <= mx[0] * 1005) best = kCands[ci];
          pdeal->phases = best;
          pdeal->items = (BH / best) * NQB;
          pdeal->rounds = (pdeal->items + G - 1) / G;
        }
      }
      fence_proxy_async_smem();  // the table's stores come before the TMA loads into the ring
    } else if (threadIdx.x == 0) {
      pdeal->phases = 1;
      pdeal->items = p.group_items;
      pdeal->rounds = p.group_rounds;
    }
    __syncthreads();
  }
  // items of this CTA, at most, and the k-th of them
  const int rounds = (PACKED && kPhased) ? pdeal->phases * pdeal->rounds : p.n_groups * p.group_rounds;
  auto next_item = [&](int k) {
    return (PACKED && kPhased) ? item_of<kPhased>(k, pdeal->items, pdeal->rounds)
                               : item_of<kPhased>(k, p.group_items, p.group_rounds);
  };
  auto wait_all = [&](uint32_t bar, uint32_t parity, unsigned site) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, p.st, abort_flag, (K_ATTN_TC << 8) | site));
  };

  if (warp == kProducerWarp) {
    // =================== TMA producer (whole warp, one elected lane issues) ===================
    // Ring loads are numbered across items (tg), so slots and phases run on.
    int tg = 0, nq = 0;
    bool ok = true;
    // Q is read once: its lines are the first to leave L2, before the K/V tiles that later items
    // read again
    const uint64_t read_once = l2_policy_evict_first();
    for (int k = 0; ok && k < rounds; ++k) {
      const int idx = next_item(k);
      if (idx < 0) continue;
      const Item it = item_at<D, PACKED, SPLIT, MODE>(p, idx, pdeal);
      if (it.n_all == 0) continue;
      // the previous item's S MMAs must have finished reading Q
      if (nq > 0 && !(ok = wait_all(bar_qempty, (uint32_t)(nq - 1) & 1u, W_QEMPTY))) break;
      mbar_arrive_expect_tx_elect(bar_q, (SPLIT ? 1 : 2) * C::Q_TILE);
      for (int i = 0; i < (SPLIT ? 1 : 2); ++i)
        for (int s = 0; s < C::SLABS; ++s)
          tma_load_3d_elect_hint(sbase + C::Q_OFF + i * C::Q_TILE + s * C::Q_SLAB, &tm_q, bar_q, s * 64,
                                 it.yq + it.q0 + i * BM, it.zq, read_once);
      ++nq;
      for (int t = 0; t < 2 * n_loads_of<SPLIT>(it); ++t, ++tg) {
        if (!(ok = wait_all(bar_empty(tg), ring_phase(tg) ^ 1u, W_KEMPTY))) break;
        mbar_arrive_expect_tx_elect(bar_full(tg), C::KV_TILE);
        const CUtensorMap* map = (t & 1) ? &tm_v : &tm_k;
        for (int s = 0; s < C::SLABS; ++s)
          tma_load_3d_elect(ring_addr(tg) + s * C::KV_SLAB, map, bar_full(tg), s * 64,
                            it.ykv + (SPLIT ? (t >> 1) : key_tile(t >> 1, it.nrev)) * C::BN, it.zkv);
      }
    }
    // drain: every load issued must have landed before the CTA can exit
    for (int t = max(0, tg - C::SLOTS); t < tg; ++t)
      mbar_wait(bar_full(t), ring_phase(t), p.st, nullptr, (K_ATTN_TC << 8) | W_DRAIN);
    if (nq > 0) mbar_wait(bar_q, (uint32_t)(nq - 1) & 1u, p.st, nullptr, (K_ATTN_TC << 8) | W_DRAIN);
  } else if (warp >= kMmaWarp0) {
    // =================== MMA issuers (whole warp, one elected lane issues) ===================
    // Descriptors are built once; per MMA only a compile-time offset is added, so every
    // operand stays warp-uniform.
    const uint64_t q_desc0 = smem_desc_sw128(sbase + C::Q_OFF, 16, 1024);
    const uint64_t k_desc0 = smem_desc_sw128(sbase + C::RING_OFF, 16, 1024);            // K: K-major
    const uint64_t v_desc0 = smem_desc_sw128(sbase + C::RING_OFF, C::KV_SLAB, 1024);  // V: MN-major
    auto slot_off = [&](int t) { return (uint64_t)(((t % C::SLOTS) * C::KV_TILE) >> 4); };
    auto issue_s = [&](int i, int t) {  // S_i = Q_i K^T (SPLIT: Q_0 for both), K from ring load t
      const uint32_t d_tmem = tmem_base + C::s_col(i);
      const uint64_t a = q_desc0 + (uint64_t)(((SPLIT ? 0 : i) * C::Q_TILE) >> 4);
      const uint64_t b = k_desc0 + slot_off(t);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t a_off = (uint64_t)(((kk / 4) * C::Q_SLAB + (kk % 4) * 32) >> 4);
        const uint64_t b_off = (uint64_t)(((kk / 4) * C::KV_SLAB + (kk % 4) * 32) >> 4);
        mma_ss_elect(d_tmem, a + a_off, b + b_off, C::IDESC_S, kk > 0 ? 1u : 0u);
      }
    };
    // O_i += P_i V over keys [16 kk0, 16 kk1) of the tile, V from ring load t
    auto issue_pv = [&](int i, int t, bool accumulate, int kk0, int kk1) {
      const uint32_t d_tmem = tmem_base + C::o_col(i);
      const uint32_t a_tmem = tmem_base + C::p_col(i);
      const uint64_t b = v_desc0 + slot_off(t);
#pragma unroll
      for (int kk = 0; kk < C::BN / 16; ++kk)
        if (kk >= kk0 && kk < kk1)
          mma_ts_elect(d_tmem, a_tmem + kk * 8, b + (uint64_t)((kk * 2048) >> 4), C::IDESC_O,
                       (accumulate || kk > 0) ? 1u : 0u);
    };
    // PV_i over the whole tile once P_i is written (with HALF_P: the first half of the keys as
    // soon as the group has written their half of P_i)
    auto wait_issue_pv = [&](int i, int t, uint32_t ph, bool accumulate) {
      constexpr int kSteps = C::BN / 16;
      if constexpr (C::HALF_P) {
        if (!wait_all(bar_phalf(i), ph, W_PFULL)) return false;
        tc_fence_after_sync();
        issue_pv(i, t, accumulate, 0, kSteps / 2);
      }
      if (!wait_all(bar_pfull(i), ph, W_PFULL)) return false;
      tc_fence_after_sync();
      issue_pv(i, t, accumulate, C::HALF_P ? kSteps / 2 : 0, kSteps);
      return true;
    };
    // Running counters across items: tg = first ring load of the item, nq = Q loads so far,
    // st_i = score tiles of query tile i so far (the phase of s_full / p_full / o_done / s_free).
    int tg = 0, nq = 0, st0 = 0, st1 = 0;
    bool ok = true;
    if constexpr (kOneIssuer) {
      // ---- one warp for both tiles: per key tile j, PV_0(j), S_0(j+1), PV_1(j), S_1(j+1) ----
      for (int k = 0; ok && k < rounds; ++k) {
        const int idx = next_item(k);
        if (idx < 0) continue;
        const Item it = item_at<D, PACKED, SPLIT, MODE>(p, idx, pdeal);
        if (it.n_all == 0) continue;
        if (!(ok = wait_all(bar_q, (uint32_t)nq & 1u, W_Q))) break;
        ++nq;
        if (!(ok = wait_all(bar_full(tg), ring_phase(tg), W_KFULL))) break;
        tc_fence_after_sync();
        for (int i = 0; i < 2; ++i)
          if (it.n_kv[i] > 0) {
            issue_s(i, tg);
            mma_commit_elect(bar_sfull(i));
          }
        mma_commit_elect(bar_empty(tg));
        if (it.n_all == 1) mma_commit_elect(bar_qempty);
        for (int j = 0; ok && j < it.n_all; ++j) {
          const int tv = tg + 2 * j + 1, tk = tg + 2 * j + 2;  // loads holding V_j and K_{j+1}
          bool k_next_ready = false;
          if (!(ok = wait_all(bar_full(tv), ring_phase(tv), W_VFULL))) break;
          for (int i = 0; i < 2 && ok; ++i) {
            if (j >= it.n_kv[i]) continue;
            if (!(ok = wait_issue_pv(i, tv, (uint32_t)((i ? st1 : st0) + j) & 1u, j > 0))) break;
            mma_commit_elect(bar_odone(i));
            if (j + 1 < it.n_kv[i]) {  // P_i lives in S_i's columns: S_i(j+1) after PV_i(j)
              if (!k_next_ready) {
                if (!(ok = wait_all(bar_full(tk), ring_phase(tk), W_KFULL))) break;
                tc_fence_after_sync();
                k_next_ready = true;
              }
              issue_s(i, tk);
              mma_commit_elect(bar_sfull(i));
            }
          }
          if (!ok) break;
          mma_commit_elect(bar_empty(tv));
          if (k_next_ready) mma_commit_elect(bar_empty(tk));
          if (j + 2 == it.n_all) mma_commit_elect(bar_qempty);  // the item's last S MMAs are issued
        }
        tg += 2 * n_loads_of<SPLIT>(it);
        st0 += it.n_kv[0];
        st1 += it.n_kv[1];
      }
    } else {
      // Each query tile's MMAs come from a warp of its own (warp 9: tile 0, warp 10: tile 1).  Per
      // tile the order follows where P_i lives: with P_i separate, S_i(j+1) as soon as the group
      // has read S_i(j), then PV_i(j); with P_i over S_i, PV_i(j) then S_i(j+1) (MMAs of one
      // thread run in issue order).
      const int i = warp - kMmaWarp0;
      auto s_next = [&](int tk, uint32_t ph, bool last_s) {  // S_i of the tile after the current one
        if (!wait_all(bar_full(tk), ring_phase(tk), W_KFULL)) return false;
        if (C::SEP_P && !wait_all(bar_sfree(i), ph, W_SFREE)) return false;
        tc_fence_after_sync();
        issue_s(i, tk);
        mma_commit_elect(bar_sfull(i));
        mma_commit_elect(bar_empty(tk));
        if (last_s) mma_commit_elect(bar_qempty);
        return true;
      };
      auto pv = [&](int tv, uint32_t ph, bool accumulate) {
        if (!wait_all(bar_full(tv), ring_phase(tv), W_VFULL)) return false;
        if (!wait_issue_pv(i, tv, ph, accumulate)) return false;
        mma_commit_elect(bar_odone(i));
        mma_commit_elect(bar_empty(tv));
        return true;
      };
      for (int k = 0; ok && k < rounds; ++k) {
        const int idx = next_item(k);
        if (idx < 0) continue;
        const Item it = item_at<D, PACKED, SPLIT, MODE>(p, idx, pdeal);
        if (it.n_all == 0) continue;
        const int n = it.n_kv[i], sb = i ? st1 : st0, n_ld = 2 * n_loads_of<SPLIT>(it);
        if (!(ok = wait_all(bar_q, (uint32_t)nq & 1u, W_Q))) break;
        ++nq;
        // Ring loads of the item: K_j in load 2j, V_j in 2j + 1.  SPLIT: slot i's m-th key tile is
        // key tile 2m + i.  The loads a tile does not read (SPLIT: the other slot's; else the other
        // tile's last key tiles) are released by a plain arrival once they have landed, in load
        // order as this warp moves past them: neither warp holds ring slots the other needs, and
        // every arrival falls in its slot's current phase.
        int rel = 0;  // loads tg + rel onwards not yet passed
        auto release_to = [&](int t_end) {
          for (; rel < t_end; ++rel) {
            const bool mine = SPLIT ? (((rel >> 1) & 1) == i) : (rel < 2 * n);
            if (mine) continue;  // read by this tile's MMAs: released by a commit
            if (!wait_all(bar_full(tg + rel), ring_phase(tg + rel), W_DRAIN)) return false;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty(tg + rel));
          }
          return true;
        };
        auto k_ld = [&](int m) { return SPLIT ? 4 * m + 2 * i : 2 * m; };  // load of the tile's m-th K
        if (n > 0) {
          if (!(ok = release_to(k_ld(0)))) break;
          if (!(ok = wait_all(bar_full(tg + k_ld(0)), ring_phase(tg + k_ld(0)), W_KFULL))) break;
          tc_fence_after_sync();
          issue_s(i, tg + k_ld(0));
          mma_commit_elect(bar_sfull(i));
          mma_commit_elect(bar_empty(tg + k_ld(0)));
          if (n == 1) mma_commit_elect(bar_qempty);
        } else {
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_qempty);  // Q(this item) has landed: the arrival is in phase
        }
        for (int m = 0; ok && m < n; ++m) {
          const int tv = tg + k_ld(m) + 1, tk = tg + k_ld(m + 1);
          const uint32_t ph = (uint32_t)(sb + m) & 1u;
          const bool more = m + 1 < n;
          if (C::SEP_P && more && !(ok = release_to(k_ld(m + 1)) && s_next(tk, ph, m + 2 == n))) break;
          if (!(ok = pv(tv, ph, m > 0))) break;
          if (!C::SEP_P && more && !(ok = release_to(k_ld(m + 1)) && s_next(tk, ph, m + 2 == n))) break;
        }
        if (ok) ok = release_to(n_ld);
        tg += n_ld;
        if (i) st1 += n; else st0 += n;
      }
    }
    {
      // drain: every MMA issued completes before TMEM is freed
      mma_commit_elect(bar_drain);
      mbar_wait(bar_drain, 0, p.st, nullptr, (K_ATTN_TC << 8) | W_DRAIN);
    }
  } else {
    // =================== softmax groups ===================
    const int i = warp >> 2;                 // query tile of this group
    const int tt = threadIdx.x & 127;        // row within the tile = TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    constexpr int BN = C::BN;
    const uint32_t s_addr = tmem_base + lane_base + C::s_col(i);
    const uint32_t o_addr = tmem_base + lane_base + C::o_col(i);
    const uint32_t p_addr = tmem_base + lane_base + C::p_col(i);
    const float sl2 = p.scale_log2;
    const uint64_t write_once = l2_policy_evict_first();
    int sb = 0;  // score tiles of this group in earlier items (barrier phases run on)
    int nx = 0;  // SPLIT: items handed over so far (the phase of xch / xdone)
    bool ok = true;
    for (int k = 0; ok && k < rounds; ++k) {
      const int idx = next_item(k);
      if (idx < 0) continue;
      // only what the score loop needs stays live through it; the epilogue looks the item up
      // again for its output offsets
      // (causal) r0 + off: the last key visible to the tile's first row; row + off: to this row's
      int n, kvl, r0, off, nrev;
      {
        const Item it = item_at<D, PACKED, SPLIT, MODE>(p, idx, pdeal);
        n = it.n_kv[i];
        nrev = it.nrev;
        kvl = it.kvl;
        r0 = it.q0 + (SPLIT ? 0 : i * BM);
        off = MODE == kCausalOff ? it.off : 0;
      }
      const int row = r0 + tt;
      // causal position of the row: its index, or its index modulo qmod when a plane's rows are the
      // queries of several heads -- at most 128 rows, so the split-slot instance (the smallest
      // position, 0, is row r0's: the tile-level test stays valid)
      const int rpos = (SPLIT && MODE == kCausalOff && p.qmod > 0) ? row % p.qmod : row;
      float m = -INFINITY;  // running max of the scaled scores, log2 units
      float l = 0.f;

      for (int j = 0; j < n; ++j) {
        const uint32_t ph = (uint32_t)(sb + j) & 1u;
        if (!(ok = wait_all(bar_sfull(i), ph, W_SFULL))) break;
        tc_fence_after_sync();
        uint32_t sr[BN];
        if constexpr (BN == 128)
          tmem_ld128(s_addr, sr);
        else
          tmem_ld32x2(s_addr, s_addr + 32, sr);
        if constexpr (C::SEP_P) {  // S_i may now be overwritten by S_i(j+1)
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_sfree(i));
        }
        float* s = reinterpret_cast<float*>(sr);
        const int col0 = (SPLIT ? 2 * j + i : key_tile(j, nrev)) * BN;  // SPLIT: this slot's j-th key tile is 2 j + i
        constexpr bool kCausalMask = MODE != kNonCausal;
        if (col0 + BN > kvl || (kCausalMask && col0 + BN - 1 > r0 + off)) {
#pragma unroll
          for (int c = 0; c < BN; ++c) {
            const int col = col0 + c;
            if (col >= kvl || (kCausalMask && col > rpos + off)) s[c] = -INFINITY;
          }
        }
        // row max of the raw scores (scale > 0 commutes with max)
        float mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[2], s[3]), mx2 = fmaxf(s[4], s[5]), mx3 = fmaxf(s[6], s[7]);
#pragma unroll
        for (int c = 8; c < BN; c += 8) {
          mx0 = max3(mx0, s[c], s[c + 1]);
          mx1 = max3(mx1, s[c + 2], s[c + 3]);
          mx2 = max3(mx2, s[c + 4], s[c + 5]);
          mx3 = max3(mx3, s[c + 6], s[c + 7]);
        }
        const float m_tile = max3(mx0, mx1, fmaxf(mx2, mx3)) * sl2;
        // Lazy rescale: keep the running reference m unless the row max grew by
        // more than kRescaleLog2 (P stays <= 2^kRescaleLog2, exact in fp32/bf16
        // range).  O and l always share the reference, so O / l is unchanged.
        const bool grow = m_tile > m + kRescaleLog2;
        const float alpha = grow ? ex2(m - m_tile) : 1.f;  // 0 when m was -inf
        if (grow) m = m_tile;
        const float ref = (m == -INFINITY) ? 0.f : m;
        const uint64_t sl2x2 = f2_pack(sl2, sl2), nref2 = f2_pack(-ref, -ref);
        uint64_t acc0 = 0, acc1 = 0;  // packed partial row sums (bit pattern 0 == {+0.f, +0.f})
        // O_i *= alpha where the reference moved.  O_i holds PV_i(j-1) by then: with P_i separate
        // the group has waited for it before writing P_i; with P_i over S_i, S_i(j) was issued after
        // PV_i(j-1) by the same thread, so that MMA finished before S_i(j) did.
        // (HALF_P: decided before the exponentials, as O_i is rescaled before the first half of P_i
        // is handed over; else at the end)
        const bool rescale = C::HALF_P && j > 0 && __any_sync(0xffffffffu, grow);
        auto rescale_o = [&]() {
          const uint64_t al2 = f2_pack(alpha, alpha);
#pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            uint32_t orr[32];
            tmem_ld32(o_addr + c, orr);
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              float o0, o1;
              f2_unpack(f2_mul(f2_pack(__uint_as_float(orr[e]), __uint_as_float(orr[e + 1])), al2), o0, o1);
              orr[e] = __float_as_uint(o0);
              orr[e + 1] = __float_as_uint(o1);
            }
            tmem_st32(o_addr + c, orr);
          }
        };
        // P = exp2(S * scale * log2 e - ref): pair c (columns 2c, 2c+1) is written as
        // one bf16x2 word into sr[c], whose scores have already been consumed.  The first half of
        // P goes to TMEM as soon as it is complete (HALF_P: O_i rescaled first, and the half handed
        // to the MMA warp at once).
        constexpr int kHalfP = BN / 4;  // words in half of P
#pragma unroll
        for (int c = 0; c < BN / 2; ++c) {
          float e0, e1;
          f2_unpack(f2_fma(f2_pack(s[2 * c], s[2 * c + 1]), sl2x2, nref2), e0, e1);
          const float p0 = ex2(e0), p1 = ex2(e1);
          if (c & 1)
            acc1 = f2_add(acc1, f2_pack(p0, p1));
          else
            acc0 = f2_add(acc0, f2_pack(p0, p1));
          sr[c] = pack_bf16x2(p0, p1);
          if (c == kHalfP - 1) {
            if (C::SEP_P && j > 0) {
              // P_i(j) goes where PV_i(j-1) reads P_i(j-1): wait for that MMA (and O_i).
              // (At j = 0 the previous item's epilogue already waited for its last PV.)
              ok = wait_all(bar_odone(i), ph ^ 1u, W_ODONE);
              tc_fence_after_sync();
            }
            if (C::HALF_P && rescale) {
              ok = wait_all(bar_odone(i), ph ^ 1u, W_ODONE);  // complete already (see rescale_o)
              tc_fence_after_sync();
              if (ok) rescale_o();
            }
            if (ok) {
              if constexpr (kHalfP == 32)
                tmem_st32(p_addr, *reinterpret_cast<const uint32_t(*)[32]>(&sr[0]));
              else
                tmem_st16(p_addr, &sr[0]);
            }
          }
          // the half is handed over a few pairs later, when its stores have (nearly) landed:
          // waiting for them at once would stall the exponentials behind the store latency
          if (C::HALF_P && c == kHalfP - 1 + kPHandoffLag && ok) {
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_phalf(i));
          }
        }
        if (!ok) break;
        if constexpr (kHalfP == 32)
          tmem_st32(p_addr + 32, *reinterpret_cast<const uint32_t(*)[32]>(&sr[32]));
        else
          tmem_st16(p_addr + 16, &sr[16]);
        float a0, a1, a2, a3;
        f2_unpack(acc0, a0, a1);
        f2_unpack(acc1, a2, a3);
        l = alpha * l + ((a0 + a1) + (a2 + a3));
        if (!C::HALF_P && j > 0 && __any_sync(0xffffffffu, grow)) rescale_o();
        tmem_st_wait();
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_pfull(i));
      }
      if (!ok) break;

      // ---- epilogue: O / l, LSE ----
      const bool have_o = n > 0;
      if (have_o && !(ok = wait_all(bar_odone(i), (uint32_t)(sb + n - 1) & 1u, W_ODONE))) break;
      tc_fence_after_sync();
      // SPLIT: the two slots hold (m, l, O) of the same rows over the even and the odd key tiles.
      // Slot 1 hands over (m, l) and its finished O_1; slot 0 merges the pairs (the reference
      // max of the two, each side rescaled to it) and writes the row; slot 1 waits until slot 0
      // has read O_1 before its next P can let PV_1 overwrite it.
      bool have_o1 = false;
      float a0 = 1.f, a1 = 0.f;
      if constexpr (SPLIT) {
        const uint32_t xph = (uint32_t)nx & 1u;
        ++nx;
        if (i == 1) {
          xch_ml[tt] = make_float2(m, have_o ? l : 0.f);
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_xch);
          if (!(ok = wait_all(bar_xdone, xph, W_ODONE))) break;
          sb += n;
          continue;
        }
        if (!(ok = wait_all(bar_xch, xph, W_ODONE))) break;
        tc_fence_after_sync();
        const float2 ml1 = xch_ml[tt];
        have_o1 = ml1.y > 0.f;
        const float mm = fmaxf(m, ml1.x);
        const float ref = (mm == -INFINITY) ? 0.f : mm;
        a0 = (m == -INFINITY) ? 0.f : ex2(m - ref);
        a1 = (ml1.x == -INFINITY) ? 0.f : ex2(ml1.x - ref);
        l = a0 * l + a1 * ml1.y;
        m = mm;
      }
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      const Item it = item_at<D, PACKED, SPLIT, MODE>(p, idx, pdeal);
      const int64_t o_rs = PACKED ? p.o_rs : D;  // O row stride
      __nv_bfloat16* orow = p.o + it.ob + (int64_t)row * o_rs;
      const bool row_in = row < it.nq && OA_DCHECK(p.st, it.ob + (int64_t)row * o_rs + D <= p.o_elems,
                                                   (K_ATTN_TC << 8) | kSiteDebugBase);
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t orr[32];
        if (have_o) {
          tmem_ld32(o_addr + c, orr);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) orr[e] = 0u;
        }
        if constexpr (SPLIT) {  // O = a0 O_0 + a1 O_1 (a side with no keys contributes nothing)
          uint32_t o1[32];
          if (have_o1) tmem_ld32(tmem_base + lane_base + C::o_col(1) + c, o1);
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float v0 = have_o ? a0 * __uint_as_float(orr[e]) : 0.f;
            orr[e] = __float_as_uint(have_o1 ? fmaf(a1, __uint_as_float(o1[e]), v0) : v0);
          }
        }
        uint4 pk[4];
        uint32_t* w = reinterpret_cast<uint32_t*>(pk);
#pragma unroll
        for (int e = 0; e < 16; ++e)
          w[e] = pack_bf16x2(__uint_as_float(orr[2 * e]) * inv_l, __uint_as_float(orr[2 * e + 1]) * inv_l);
        // Each thread writes its own row: a warp's store touches 32 rows, so whole 32-byte
        // sectors per thread (half as many requests as 16-byte stores) matter here.
        if (row_in) {
          if (p.o_v8) {  // O is written once: first out of L2 (see the Q loads)
            st_global_v8_hint(orow + c, w, write_once);
            st_global_v8_hint(orow + c + 16, w + 8, write_once);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(orow + c);
            dst[0] = pk[0];
            dst[1] = pk[1];
            dst[2] = pk[2];
            dst[3] = pk[3];
          }
        }
      }
      if (p.lse != nullptr && row < it.nq &&
          OA_DCHECK(p.st, it.lb + (int64_t)row * (PACKED ? p.l_rs : 1) < p.lse_elems, (K_ATTN_TC << 8) | (kSiteDebugBase + 1)))
        p.lse[it.lb + (int64_t)row * (PACKED ? p.l_rs : 1)] = (l > 0.f) ? (m + log2f(l)) * kLn2 : -INFINITY;
      // O_i has been read out: the next item's PV_i(0) (issued after this group's next P)
      // may overwrite it
      tc_fence_before_sync();
      if constexpr (SPLIT) {  // and O_1 and slot 1's (m, l) too
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_xdone);
      }
      sb += n;
    }
  }

  // ---- teardown ----
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

constexpr int kMaxDevices = 64;

// Dealing of a dense causal launch on G CTAs (see item_of).  When the K/V of the launch does not
// fit in L2, either (key offset, items of nearly equal weight) the items are numbered plane by
// plane, or the heads are split into bands of whole key/value planes swept one after the other
// in phases; either way the items running at the same time read the K/V of few planes.  The phase
// count is the largest of 2, 4 and 8 whose dealing leaves the busiest CTA at most 0.5 % busier
// than one phase does, and the plane-by-plane numbering is taken when the lightest item weighs
// at least 0.9 of the heaviest and its dealing leaves the busiest CTA at most 0.2 % busier
// (chunked prefill B8 H32 H_kv 8, 2048 queries after 30720 cached keys: +0.8 %; at B2, 0.4 %
// busier in the simulation, it measured 0.8 % slower) (weights: the key tiles an item loads plus
// two for its Q load and epilogue; kv_len, unknown here, is taken as Nk).  The choice is kept per
// shape.
struct Dealing {
  int phases, plane_major;
};
template <int D, int MODE>
Dealing causal_dealing(const TcParams& p, int G) {
  constexpr int BN = Cfg<D>::BN;
  constexpr long long kL2Bytes = 48ll << 20;  // K/V that stays in L2 through a phase
  const int planes = p.BH / p.group;
  const long long kv_bytes = (long long)planes * p.Nk * D * 2 * 2;
  const long long total = (long long)p.num_qblocks * p.BH;
  if (kv_bytes <= kL2Bytes || total > (1 << 16) || G < 1) return Dealing{1, 0};
  struct Entry { int nqb, bh, group, nq, nk, off, G; Dealing d; };
  thread_local Entry cache[4] = {};
  thread_local int next = 0;
  const int off = MODE == kCausalOff ? p.off : 0;
  for (const Entry& c : cache)
    if (c.d.phases > 0 && c.nqb == p.num_qblocks && c.bh == p.BH && c.group == p.group && c.nq == p.Nq &&
        c.nk == p.Nk && c.off == off && c.G == G)
      return c.d;
  // weight of an item of query block qb (both query tiles share its key tiles)
  std::vector<long long> w(p.num_qblocks);
  const int nk_tiles = (p.Nk + BN - 1) / BN;
  for (int qb = 0; qb < p.num_qblocks; ++qb) {
    int n = 0;
    for (int i = 0; i < 2; ++i) {
      const int r0 = qb * 2 * BM + i * BM;
      if (r0 < p.Nq) n = std::max(n, std::max(0, std::min(nk_tiles, (r0 + BM - 1 + off + BN) / BN)));
    }
    w[qb] = n + 2;
  }
  std::vector<long long> load(G);
  auto busiest = [&](int ng, bool by_plane) {
    const int hs = p.BH / ng, gi = hs * p.num_qblocks, gr = (gi + G - 1) / G;
    std::fill(load.begin(), load.end(), 0ll);
    for (int f = 0; f < ng; ++f)
      for (int kr = 0; kr < gr; ++kr)
        for (int b = 0; b < G; ++b) {
          const int c = (f & 1) ? G - 1 - b : b;
          const int r = kr * G + ((kr & 1) ? (G - 1 - c) : c);
          if (r < gi) load[b] += w[p.num_qblocks - 1 - (by_plane ? r % p.num_qblocks : r / hs)];
        }
    return *std::max_element(load.begin(), load.end());
  };
  const long long one = busiest(1, false);
  Dealing best{1, 0};
  const long long w_min = *std::min_element(w.begin(), w.end()), w_max = *std::max_element(w.begin(), w.end());
  if (MODE == kCausalOff && 10 * w_min >= 9 * w_max && (double)busiest(1, true) <= 1.002 * (double)one) {
    best.plane_major = 1;
  } else {
    for (int ng = 2; ng <= 8; ng *= 2)
      if (planes % ng == 0 && (double)busiest(ng, false) <= 1.005 * (double)one) best.phases = ng;
  }
  cache[next] = Entry{p.num_qblocks, p.BH, p.group, p.Nq, p.Nk, off, G, best};
  next = (next + 1) % 4;
  return best;
}

// Persistent grid: one CTA per SM (the kernel holds an SM's TMEM and most of its shared
// memory), never more CTAs than work items.  Without the causal mask (and without packed
// sequences) the items weigh alike, so the grid is the fewest CTAs that keep the number of rounds:
// every CTA then works through the same number of items, and the memory-bound cases (grouped
// decode) spread the same bytes over fewer, busier CTAs instead of a last round half empty.
template <int D, bool PACKED, bool SPLIT, int MODE>
cudaError_t launch_d(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv, const TcParams& p,
                     cudaStream_t s) {
  static bool attr_set[kMaxDevices] = {};
  static int sm_count[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(attn_fwd_tc_kernel<D, PACKED, SPLIT, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg<D>::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const long long total = (long long)p.num_qblocks * p.BH;
  long long g = total < sm_count[dev] ? total : sm_count[dev];
  if (!PACKED && MODE == kNonCausal) {
    const long long rounds = (total + g - 1) / g;
    g = (total + rounds - 1) / rounds;
  }
  TcParams q = p;
  // (packed: one phase here; the kernel may choose more, see PackedDeal)
  const Dealing deal = (phased<PACKED, SPLIT, MODE>() && !PACKED) ? causal_dealing<D, MODE>(p, (int)g)
                                                                   : Dealing{1, 0};
  q.n_groups = deal.phases;
  q.plane_major = deal.plane_major;
  q.group_items = (int)(total / q.n_groups);
  q.group_rounds = (int)((q.group_items + g - 1) / g);
  q.dir_hs = q.BH / q.n_groups;
  q.dir_G = (int)g;
  q.dir_sh0 = 0;
  q.dir_alt = !deal.plane_major;  // a plane's items read its K/V together, in step
  if (phased<PACKED, SPLIT, MODE>() && p.call_bh > p.BH) {  // a piece of a call of call_bh planes
    TcParams whole = p;
    whole.BH = p.call_bh;
    const long long total_w = (long long)p.num_qblocks * whole.BH;
    const long long g_w = total_w < sm_count[dev] ? total_w : sm_count[dev];
    const Dealing dw = causal_dealing<D, MODE>(whole, (int)g_w);
    q.dir_hs = whole.BH / dw.phases;
    q.dir_G = (int)g_w;
    q.dir_sh0 = p.call_sh0;
    q.dir_alt = !dw.plane_major;
  }
  const unsigned grid = (unsigned)g;
  attn_fwd_tc_kernel<D, PACKED, SPLIT, MODE><<<grid, Cfg<D>::template threads<SPLIT>(), Cfg<D>::SMEM_BYTES, s>>>(mq, mk, mv, q);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_tc(const TcArgs& a, const DevStatus& st, cudaStream_t s, const char** why) {
  const int d = a.d, Hkv = a.Hkv;
  const bool packed = a.cu_q != nullptr;
  const int64_t rb = 2 * (int64_t)d;  // bytes per row of one head
  const int kv_rows = d == 128 ? Cfg<128>::BN : Cfg<64>::BN;  // key/value tile height (TMA box)
  CUtensorMap mq, mk, mv;
  bool maps_ok;
  if (packed)
    maps_ok = make_tile_map(&mq, a.q, d, a.Tq, rb * a.H, a.H, rb, BM) &&
              make_tile_map(&mk, a.k, d, a.Tk, rb * Hkv, Hkv, rb, kv_rows) &&
              make_tile_map(&mv, a.v, d, a.Tk, rb * Hkv, Hkv, rb, kv_rows);
  else
    maps_ok = make_tile_map(&mq, a.q, d, a.Nq, rb, a.B * a.H, rb * a.Nq, BM) &&
              make_tile_map(&mk, a.k, d, a.Nk, rb, a.B * Hkv, rb * a.Nk, kv_rows) &&
              make_tile_map(&mv, a.v, d, a.Nk, rb, a.B * Hkv, rb * a.Nk, kv_rows);
  if (!maps_ok) {
    if (why) *why = "cuTensorMapEncodeTiled failed or is unavailable";
    return cudaErrorInvalidValue;
  }
  TcParams p;
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.o_v8 = (reinterpret_cast<uintptr_t>(a.o) % 32u) == 0 ? 1 : 0;
  p.lse = a.lse;
  p.kv_len = packed ? nullptr : a.kv_len;
  p.cu_q = a.cu_q;
  p.cu_k = a.cu_k;
  p.Tq = a.Tq;
  p.Tk = a.Tk;
  p.H = a.H;
  p.Nq = a.Nq;
  p.Nk = a.Nk;
  p.off = a.Nk - (a.qmod > 0 ? a.qmod : a.Nq);
  p.qmod = a.qmod;
  p.num_qblocks = (a.Nq + 2 * BM - 1) / (2 * BM);
  p.BH = a.B * a.H;
  p.group = a.H / Hkv;
  p.o_rs = packed ? (int64_t)a.H * d : d;
  p.o_elems = packed ? (int64_t)a.Tq * a.H * d : (int64_t)a.B * a.H * a.Nq * d;
  p.lse_elems = packed ? (int64_t)a.Tq * a.H : (int64_t)a.B * a.H * a.Nq;
  p.l_rs = packed ? a.H : 1;
  p.scale_log2 = a.scale * kLog2e;
  p.st = st;
  // packed causal with more K/V than L2 keeps: the kernel decides its phases (see PackedDeal)
  p.decide_phases = (packed && a.causal && (long long)a.Tk * Hkv * d * 4 > (48ll << 20)) ? 1 : 0;
  p.call_bh = (!packed && a.order_bh > p.BH) ? a.order_bh : p.BH;
  p.call_sh0 = (!packed && a.order_bh > p.BH) ? a.order_sh0 : 0;
  if ((long long)p.num_qblocks * p.BH == 0) return cudaSuccess;  // no query rows
  // Instance by layout, query-tile use and masking mode (packed sequences may each have their own
  // key offset; a dense call has one, Nk - Nq)
  const int mode = !a.causal ? kNonCausal : (packed || a.qmod > 0 || a.Nk != a.Nq) ? kCausalOff : kCausal;
  if (packed) {
    if (mode == kNonCausal)
      return d == 128 ? launch_d<128, true, false, kNonCausal>(mq, mk, mv, p, s)
                      : launch_d<64, true, false, kNonCausal>(mq, mk, mv, p, s);
    return d == 128 ? launch_d<128, true, false, kCausalOff>(mq, mk, mv, p, s)
                    : launch_d<64, true, false, kCausalOff>(mq, mk, mv, p, s);
  }
  // At most 128 query rows (decode, multi-token decode against a cache, and grouped decode whose
  // group's queries are the rows): an item fills only one query-tile slot, so both slots take the
  // same rows over alternate key tiles and their results are merged (see item_at).  A square
  // causal call this small runs as the offset mode with offset 0.
  if (a.Nq <= BM) {
    if (mode == kNonCausal)
      return d == 128 ? launch_d<128, false, true, kNonCausal>(mq, mk, mv, p, s)
                      : launch_d<64, false, true, kNonCausal>(mq, mk, mv, p, s);
    return d == 128 ? launch_d<128, false, true, kCausalOff>(mq, mk, mv, p, s)
                    : launch_d<64, false, true, kCausalOff>(mq, mk, mv, p, s);
  }
  if (mode == kNonCausal)
    return d == 128 ? launch_d<128, false, false, kNonCausal>(mq, mk, mv, p, s)
                    : launch_d<64, false, false, kNonCausal>(mq, mk, mv, p, s);
  if (mode == kCausal)
    return d == 128 ? launch_d<128, false, false, kCausal>(mq, mk, mv, p, s)
                    : launch_d<64, false, false, kCausal>(mq, mk, mv, p, s);
  return d == 128 ? launch_d<128, false, false, kCausalOff>(mq, mk, mv, p, s)
                  : launch_d<64, false, false, kCausalOff>(mq, mk, mv, p, s);
}

}  // namespace oa
