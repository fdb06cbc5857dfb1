// Paged prefill on the 5th-generation tensor cores (tcgen05.mma, TMEM).
//
// What it computes is the prefill of prefill.cu ("Make the Engine Talk",
// 1.2: one forward pass over all of a prompt's tokens, which fills the KV
// cache): query token i of sequence b's run of n_b tokens sits at position
// p = L_b - n_b + i and attends to every cached position t <= p of its KV
// head's group.
//
// One CTA per SM-sized piece of work: a pair of query tiles of the same
// (sequence, KV head g).  A query tile is M = 128 MMA rows: 128 / G
// consecutive query tokens x the G heads of group g (row r is token r / G,
// head g*G + r % G); the second tile holds the next 128 / G tokens.  Both
// tiles read the same K/V stream, so each K/V byte crosses from L2 once per
// 256 query rows.  Ten warps with fixed roles:
//   * warp 8 (producer) loads the two Q tiles once (3-D TMA boxes of 64 dims
//     x G heads x 128/G tokens, which land as 128 K-major rows each) and
//     streams the sequence's K and V, 128 tokens (8 blocks) per stage,
//     through the block table into a 2-stage K ring and a 3-stage V ring, up
//     to the pair's last query position.  K(j) and V(j) are requested as
//     soon as their slots free; V's slot frees later (after both P V of a
//     stage, where K's frees after both Q K^T), so V gets the deeper ring.
//     Block ids are read 32 at a time (four stages), a group ahead, and
//     lane u issues block u's boxes: issued from one thread, a half-stage's
//     16 boxes took longer than the MMAs that read them;
//   * warp 9 (MMA) owns all 512 TMEM columns: O_0, O_1 (D columns each at
//     0 and 128) and S_0, S_1 (128 columns each at 256 and 384).  Its lane 0
//     issues S_t = Q_t K_j^T (M 128, N 128, K = D; both operands K-major in
//     shared memory as TMA wrote them) and O_t += P_t V_j (M 128, N = D,
//     K 128; P from TMEM over S_t, V MN-major as it lies in the stage).  The
//     order PV_0(j), QK_0(j+1), PV_1(j), QK_1(j+1) keeps one tile's MMAs
//     running while the other tile's softmax works; each P V runs in two
//     halves of 64 tokens, the first as soon as the softmax has written
//     those tokens' weights.  S_t is rewritten only after the P_t V that
//     reads it has completed (tcgen05.commit on mbarriers tracks completion
//     and frees stages);
//   * warps 0-3 and 4-7 are the softmax warpgroups of tiles 0 and 1: one row
//     per thread, warp w reading TMEM lanes 32 (w % 4) .. +31.  Per stage:
//     load the row of S, mask by position (only on stages that reach past
//     the row's position), and keep a running maximum that moves only when
//     the row's maximum grows by more than 8 in log2 units, so the weights
//     stay <= 2^8 and O is rescaled rarely (O_t is idle then: the previous
//     P_t V has completed before S_t was written).  The row is read twice
//     from TMEM, for its maximum and then 64 tokens at a time for the
//     weights (the second 64 while the first 64's weights are stored), which
//     keeps the registers of 320 threads within the SM.  The
//     weights P = 2^(scale s - m) go over the 32 columns of S they came from,
//     as bf16 high parts (16 columns, two weights per column) and low parts
//     (the next 16), so P V keeps ~16 bits of each weight: a weight rounded
//     to bf16 once could move a bf16 output by as much as its own rounding.
//     At the end O is divided by the row sum and stored.
// Shared memory is 225 KB (D = 128) and TMEM 512 columns, one CTA per SM.
// V rows that may hold anything (the tail of the last block, or blocks the
// last stage did not load) are zeroed before P V reads them: P is 0 there,
// but 0 * NaN is NaN.  Every mbarrier wait is bounded; the MMA warp drains
// its own MMAs before TMEM is freed.
#include <atomic>

#include "common.cuh"
#include "tcgen05.cuh"

namespace forge {
namespace {

constexpr int kTcRows = 128;                 // MMA M: rows of one query tile
constexpr int kTcTiles = 2;                  // query tiles per CTA
constexpr int kTcKv = 128;                   // tokens per K/V stage (MMA N of S, K of P V)
constexpr int kTcKStages = 2;                // K ring depth
constexpr int kTcVStages = 3;                // V ring depth
constexpr int kTcSoftmaxWarps = 4 * kTcTiles;
constexpr int kTcProducerWarp = kTcSoftmaxWarps;
constexpr int kTcMmaWarp = kTcSoftmaxWarps + 1;
constexpr int kTcThreads = (kTcSoftmaxWarps + 2) * 32;
constexpr int kTmemCols = 512;
constexpr int kColO = 0;                     // O_t at kColO + 128 t (D columns)
constexpr int kColS = 256;                   // S_t (and P_t over it) at kColS + 128 t
constexpr float kRescaleSlack = 8.0f;        // log2 units: weights stay <= 2^8
constexpr unsigned kFullMask = 0xffffffffu;
constexpr int kMinSmem = 116 * 1024;         // > half an SM's shared memory: one CTA per SM
static_assert(kTcTiles * kTcRows == kPrefillChunkRows, "partial rows of a chunk");

struct TcLayout {
  int q, k, v, bars, total;
};

// Q [tile][box][128 rows][128 B] | K ring [stage][box][128 tok][128 B] |
// V ring (same) | mbarriers, TMEM slot.  Offsets from a 1024-byte-aligned base.
// Whether the phase of `bar` with this parity has completed, without waiting
// (acquire semantics when it has).
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__host__ __device__ constexpr int q_tile_bytes(int D) { return (D / 64) * kTcRows * 128; }
__host__ __device__ constexpr int kv_stage_bytes(int D) { return (D / 64) * kTcKv * 128; }
__host__ __device__ constexpr TcLayout tc_layout(int D) {
  TcLayout l{};
  l.q = 0;
  l.k = kTcTiles * q_tile_bytes(D);
  l.v = l.k + kTcKStages * kv_stage_bytes(D);
  l.bars = l.v + kTcVStages * kv_stage_bytes(D);
  const int used = l.bars + 32 * 8 + 1024;   // barriers + slot, + alignment slack
  l.total = used > kMinSmem ? used : kMinSmem;
  return l;
}

// mbarrier slots
constexpr int kQFull = 0;
constexpr int kKFull = 1;                       // [kTcKStages]
constexpr int kKEmpty = kKFull + kTcKStages;    // [kTcKStages]: both S = Q K^T of the stage done
constexpr int kVFull = kKEmpty + kTcKStages;    // [kTcVStages]
constexpr int kVEmpty = kVFull + kTcVStages;    // [kTcVStages]: both P V of the stage done
constexpr int kSFull = kVEmpty + kTcVStages;    // [kTcTiles]: S_t(j) written
constexpr int kPFull = kSFull + kTcTiles;     // [kTcTiles]: P_t(j) written (one arrival per softmax warp)
constexpr int kPvDone = kPFull + kTcTiles;    // [kTcTiles]: P_t(j) V_j done
constexpr int kDrain = kPvDone + kTcTiles;
constexpr int kPHalf = kDrain + 1;            // [kTcTiles]: P_t(j)'s first half written (one arrival per softmax warp)
constexpr int kSlot = kPHalf + kTcTiles;      // TMEM address (4 bytes) after the barriers

// 32 consecutive outputs of a row: fp32 accumulators times `inv`.
__device__ __forceinline__ void store_row32(float* dst, const uint32_t (&v)[32], float inv) {
#pragma unroll
  for (int c = 0; c < 32; c += 4)
    *reinterpret_cast<float4*>(dst + c) = make_float4(__uint_as_float(v[c]) * inv, __uint_as_float(v[c + 1]) * inv,
                                                      __uint_as_float(v[c + 2]) * inv, __uint_as_float(v[c + 3]) * inv);
}
__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const uint32_t (&v)[32], float inv) {
#pragma unroll
  for (int c = 0; c < 32; c += 8) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      w[e] = pack_bf16x2(__uint_as_float(v[c + 2 * e]) * inv, __uint_as_float(v[c + 2 * e + 1]) * inv);
    *reinterpret_cast<uint4*>(dst + c) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Find (sequence, first query token) of work item `tile_id` (QT query tokens
// each) from query_start: a warp scan over the sequences' item counts, the
// same answer in every warp.  Items are numbered by sequence, then by
// position in the run.
template <int QT>
__device__ __forceinline__ void find_tile(const PrefillParams& p, int tile_id, int lane, int& b, int& i0) {
  b = -1;
  i0 = 0;
  int base = 0;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    const int bb = b0 + lane;
    int nt = 0;
    if (bb < p.B) {
      const int n = __ldg(p.query_start + bb + 1) - __ldg(p.query_start + bb);
      nt = n > 0 ? (n + QT - 1) / QT : 0;
    }
    int incl = nt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(kFullMask, incl, off);
      if (lane >= off) incl += v;
    }
    const int total = __shfl_sync(kFullMask, incl, 31);
    if (tile_id < base + total) {
      const int first = __ffs(__ballot_sync(kFullMask, tile_id < base + incl)) - 1;
      const int before = __shfl_sync(kFullMask, incl - nt, first);
      b = b0 + first;
      i0 = (tile_id - base - before) * QT;
      return;
    }
    base += total;
  }
}

// The work item at place k of a longest-first order (k = 0 runs first): a
// work item's cost grows with the context it attends to, so items go by
// sequence length (longest first, ties by sequence index), and within a
// sequence from its last item to its first.  Every CTA derives the order
// from the lengths (O(B^2 / 32) loads per warp, so only for B <= kLptMaxB;
// larger batches keep the order of find_tile, reversed).
constexpr int kLptMaxB = 256;
template <int QT>
__device__ __forceinline__ void find_tile_lpt(const PrefillParams& p, int k, int lane, int& b, int& i0) {
  b = -1;
  i0 = 0;
  auto items = [&](int s) {
    const int n = __ldg(p.query_start + s + 1) - __ldg(p.query_start + s);
    return n > 0 ? (n + QT - 1) / QT : 0;
  };
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    const int bb = b0 + lane;
    int before = 0, nt = 0;
    if (bb < p.B) {
      nt = items(bb);
      const int Lb = __ldg(p.context_lens + bb);
      // items of every sequence that comes before bb in the order
      for (int s = 0; s < p.B; ++s) {
        const int Ls = __ldg(p.context_lens + s);
        if (Ls > Lb || (Ls == Lb && s < bb)) before += items(s);
      }
    }
    const bool mine = bb < p.B && k >= before && k < before + nt;
    const unsigned who = __ballot_sync(kFullMask, mine);
    if (who) {
      const int src = __ffs(who) - 1;
      b = b0 + src;
      const int idx = k - __shfl_sync(kFullMask, before, src);
      i0 = (__shfl_sync(kFullMask, nt, src) - 1 - idx) * QT;  // the sequence's last item first
      return;
    }
  }
}

template <int D, int G, typename OutT>
__global__ void __launch_bounds__(kTcThreads, 1)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                            const __grid_constant__ CUtensorMap tmv, const PrefillParams p) {
  constexpr int QT = kTcRows / G;            // query tokens per tile
  constexpr int QT2 = kTcTiles * QT;         // per CTA
  constexpr int BOXES = D / 64;
  constexpr int KSTEPS = D / 16;             // K steps of S = Q K^T
  constexpr int PSTEPS = kTcKv / 16;         // K steps of O += P V
  constexpr TcLayout lay = tc_layout(D);
  constexpr int QTILE = q_tile_bytes(D);
  constexpr int STAGE = kv_stage_bytes(D);   // 128 tokens of K (or V)
  constexpr uint32_t IDESC_S = tc::idesc_bf16_f32(kTcRows, kTcKv, false);
  constexpr uint32_t IDESC_O = tc::idesc_bf16_f32(kTcRows, D, true);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // One-dimensional grid, the KV head fastest, then the chunk slot: CTA k
  // runs chunk slot (k / Hkv) % max_chunks of work item k / (Hkv max_chunks)
  // of the longest-first order, for KV head k % Hkv, so the order holds
  // across the heads too (the hardware dispatches CTAs by increasing index).
  const int chunk_slots = max(1, p.max_chunks);
  const int g = static_cast<int>(blockIdx.x % static_cast<unsigned>(p.Hkv));
  const int unit = static_cast<int>(blockIdx.x / static_cast<unsigned>(p.Hkv));
  const int item = unit / chunk_slots, cslot = unit % chunk_slots;
  const int items = static_cast<int>(gridDim.x / static_cast<unsigned>(p.Hkv)) / chunk_slots;
  const int tile_id = items - 1 - item;  // later (longer) work first

  // query_start must start at 0, never decrease and end within the T rows
  if (blockIdx.x == 0 && warp == 0) {
    bool bad = lane == 0 && __ldg(p.query_start) != 0;
    for (int b = lane; b < p.B; b += 32) {
      const int s0 = __ldg(p.query_start + b), s1 = __ldg(p.query_start + b + 1);
      bad |= s1 < s0 || s1 > p.T;
    }
    if (__any_sync(kFullMask, bad) && lane == 0) record_error(p.err, kDevErrQuery);
  }

  int b, i0;
  if (p.B <= kLptMaxB)
    find_tile_lpt<QT2>(p, item, lane, b, i0);
  else
    find_tile<QT2>(p, tile_id, lane, b, i0);
  if (b < 0) return;  // past the last work item

  const int q0 = __ldg(p.query_start + b);
  const int n = __ldg(p.query_start + b + 1) - q0;
  const int L = __ldg(p.context_lens + b);
  if (L < 0 || L > p.MB * kBlockSize || n > L || q0 < 0 || q0 + n > p.T) {
    if (threadIdx.x == 0) record_error(p.err, (L < 0 || L > p.MB * kBlockSize) ? kDevErrLength : kDevErrQuery);
    return;
  }
  const int pos0 = L - n + i0;                     // position of the CTA's first query token
  const int p_max = pos0 + min(QT2, n - i0) - 1;   // of its last (<= L - 1)
  const int nkv_all = p_max / kTcKv + 1;           // the item's stages, up to and including p_max
  // Context chunks, aligned to the end: chunk nch-1 ends at stage nkv_all-1,
  // every chunk but chunk 0 holds C stages and chunk 0 the remaining 1..C.
  // Chunk slot c runs chunk nch-1-c (the full chunks first).  Every chunk's
  // first stage starts at or before the item's first query position, so
  // each row sees a token in it and its running maximum is finite from there.
  const int C = p.chunk_stages;
  const int nch = C > 0 ? (nkv_all + C - 1) / C : 1;
  if (cslot >= nch) return;                        // an empty chunk slot
  const int ch = nch - 1 - cslot;
  const int rem = nkv_all - (nch - 1) * (C > 0 ? C : 0);
  const int st0 = ch == 0 ? 0 : rem + (ch - 1) * C;  // this CTA's first stage
  const int nkv = ch == 0 ? rem : C;                 // and its stage count

  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                       ~static_cast<uintptr_t>(1023));
  const uint32_t sm_s = smem_addr(sm);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + lay.bars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kSlot);

  if (threadIdx.x == 0) {
    mbar_init(bars + kQFull, 1);
    for (int i = 0; i < kTcKStages; ++i) {
      mbar_init(bars + kKFull + i, 1);
      mbar_init(bars + kKEmpty + i, 1);
    }
    for (int i = 0; i < kTcVStages; ++i) {
      mbar_init(bars + kVFull + i, 1);
      mbar_init(bars + kVEmpty + i, 1);
    }
    for (int t = 0; t < kTcTiles; ++t) {
      mbar_init(bars + kSFull + t, 1);
      mbar_init(bars + kPFull + t, 4);   // one arrival per softmax warp of the tile
      mbar_init(bars + kPHalf + t, 4);
      mbar_init(bars + kPvDone + t, 1);
    }
    mbar_init(bars + kDrain, 1);
    fence_barrier_init();
  }
  if (warp == kTcMmaWarp) {
    tc::tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == kTcProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(bars + kQFull, kTcTiles * QTILE);
#pragma unroll
      for (int t = 0; t < kTcTiles; ++t)
#pragma unroll
        for (int c = 0; c < BOXES; ++c)
          tma_load_3d(sm + lay.q + t * QTILE + c * kTcRows * 128, &tmq, c * 64, g * G, q0 + i0 + t * QT,
                      bars + kQFull);
    }
    const int32_t* row = p.block_tables + static_cast<int64_t>(b) * p.bt_sb;
    constexpr int BPS = kTcKv / kBlockSize;  // blocks per stage (8)
    constexpr int GRP = 32 / BPS;            // stages per warp-wide table read (4)
    // Block ids of stages GRP q .. GRP q + GRP - 1: lane l holds block l % BPS
    // of stage GRP q + l / BPS (entries past p_max's block are not read)
    auto table_group = [&](int q) -> int {
      const int jb = BPS * (st0 + GRP * q) + lane;
      return jb * kBlockSize <= p_max ? __ldg(row + jb) : -1;
    };
    // One half (K or V) of stage j, its block ids `grp` (the group holding
    // stage j): wait for its ring slot, then one TMA box per block and 64
    // dims (blocks past p_max's block are not loaded).
    auto load_half = [&](int j, bool is_v, int grp) {
      const int jb = BPS * (st0 + j) + lane;  // j: this CTA's stage index
      const bool used = lane < BPS && jb * kBlockSize <= p_max;
      const int eg = __shfl_sync(kFullMask, grp, (j % GRP) * BPS + (lane % BPS));
      int e = used ? eg : -1;
      const bool bad = used && static_cast<unsigned>(e) >= static_cast<unsigned>(p.NB);
      if (bad) e = -1;
      if (__any_sync(kFullMask, bad) && lane == 0 && !is_v) record_error(p.err, kDevErrBlockId);
      const int nvalid = __popc(__ballot_sync(kFullMask, e >= 0));
      const int depth = is_v ? kTcVStages : kTcKStages;
      const int st = j % depth, use = j / depth;
      uint64_t* full = bars + (is_v ? kVFull : kKFull) + st;
      uint64_t* empty = bars + (is_v ? kVEmpty : kKEmpty) + st;
      unsigned char* dst = sm + (is_v ? lay.v : lay.k) + st * STAGE;
      // the whole warp waits for the slot, released by the MMAs that read it
      if (use > 0) mbar_wait(empty, (use - 1) & 1, p.err);
      if (lane == 0) {
        if (nvalid > 0)
          mbar_arrive_expect_tx(full, static_cast<uint32_t>(nvalid) * BOXES * kBlockSize * 128);
        else
          mbar_arrive(full);  // nothing to copy (a bad id is recorded above)
      }
      __syncwarp();
      // lane u < BPS copies block u: eight issuing threads, not one
      if (e >= 0) {
#pragma unroll
        for (int c = 0; c < BOXES; ++c)
          tma_load_4d(dst + c * kTcKv * 128 + lane * kBlockSize * 128, is_v ? &tmv : &tmk, c * 64, 0, g, e, full);
      }
    };
    // K(j) then V(j): each waits only for its own slot, released by QK^T of
    // stage j - 2 (K) or P V of stage j - 3 (V).  The block ids are read a
    // group of stages ahead, so no table read waits in this loop.
    int cur = table_group(0), nxt = nkv > GRP ? table_group(1) : -1;
    for (int j = 0; j < nkv; ++j) {
      if (j > 0 && j % GRP == 0) {
        cur = nxt;
        nxt = j + GRP < nkv ? table_group(j / GRP + 1) : -1;
      }
      load_half(j, false, cur);
      load_half(j, true, cur);
    }
  } else if (warp == kTcMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    // Pipe order PV_0(j), QK_0(j+1), PV_1(j), QK_1(j+1): while tile t's
    // softmax turns S_t(j+1) into weights, the other tile's MMAs run.  The
    // whole warp runs the loop and its waits, converged; lane 0's instance of
    // each MMA and commit runs (a predicate inside the instruction), so one
    // thread issues them all and each commit tracks all of them.  (Issued
    // under a lane-0 branch, beside the softmax warps, the MMAs took ~84
    // cycles each, against the 64 one runs.)
    // The descriptors are built once: the start address of a shared-memory
    // operand sits in a descriptor's low 14 bits (address >> 4, all of this
    // CTA's shared memory fits), so the tile, the ring slot and the K step
    // are added to the built descriptor as offsets >> 4.
    const uint64_t dq0 = tc::smem_desc_sw128(sm_s + lay.q, 0, 1024);
    const uint64_t dk0 = tc::smem_desc_sw128(sm_s + lay.k, 0, 1024);
    const uint64_t dv0 = tc::smem_desc_sw128(sm_s + lay.v, kTcKv * 128, 1024);
    auto issue_qk = [&](int t, int j) {
      const uint64_t dq = dq0 + static_cast<uint32_t>((t * QTILE) >> 4);
      const uint64_t dk = dk0 + static_cast<uint32_t>(((j % kTcKStages) * STAGE) >> 4);
      const uint32_t ds = tmem + kColS + kTcRows * t;
#pragma unroll
      for (int k = 0; k < KSTEPS; ++k) {
        // box of 64 dims, then the 16-dim step inside its 128-byte rows
        tc::mma_bf16_ss_lane0(ds, dq + (((k >> 2) * kTcRows * 128 + (k & 3) * 32) >> 4),
                              dk + (((k >> 2) * kTcKv * 128 + (k & 3) * 32) >> 4), IDESC_S, k > 0);
      }
      tc::commit_lane0(smem_addr(bars + kSFull + t));
      if (t == kTcTiles - 1) tc::commit_lane0(smem_addr(bars + kKEmpty + j % kTcKStages));  // both S of stage j issued
    };
    bool ok = mbar_wait(bars + kQFull, 0, p.err);
    if (ok) ok = mbar_wait(bars + kKFull + 0, 0, p.err);
    ok = __all_sync(kFullMask, ok);
    if (ok) {
      tc::fence_after_sync();
      issue_qk(0, 0);
      issue_qk(1, 0);
    }
    for (int j = 0; ok && j < nkv; ++j) {
      const int sv = j % kTcVStages;
      const uint64_t dv = dv0 + static_cast<uint32_t>((sv * STAGE) >> 4);
      for (int t = 0; ok && t < kTcTiles; ++t) {
        // P over S_t: K step kk (16 tokens) is in chunk kk / 2 (32 columns):
        // high parts at 32 (kk / 2) + 8 (kk % 2), low parts 16 columns on.
        // The first half of the K steps runs once the softmax has written the
        // first 64 tokens' weights, while it computes the rest; when all of
        // P_t is already written, all of them go out at once.  V_j has landed
        // by then: tile 0's softmax warps wait for it before their first
        // arrival of the stage.
        const uint32_t pcol = tmem + kColS + kTcRows * t, dout = tmem + kColO + kTcRows * t;
        const bool whole = __all_sync(kFullMask, mbar_test(bars + kPFull + t, j & 1));
        if (whole) tc::fence_after_sync();
        for (int half = 0; ok && half < 2; ++half) {
          if (!whole) {
            ok = mbar_wait(bars + (half == 0 ? kPHalf : kPFull) + t, j & 1, p.err);
            ok = __all_sync(kFullMask, ok);
            if (!ok) break;
            tc::fence_after_sync();
          }
#pragma unroll
          for (int k2 = 0; k2 < PSTEPS / 2; ++k2) {
            const int kk = half * (PSTEPS / 2) + k2;
            const uint32_t phi = pcol + 32 * (kk >> 1) + 8 * (kk & 1);
            const uint64_t bd = dv + ((kk * 16 * 128) >> 4);  // 16 token rows of 128 bytes
            tc::mma_bf16_ts_lane0(dout, phi, bd, IDESC_O, j > 0 || kk > 0);
            tc::mma_bf16_ts_lane0(dout, phi + 16, bd, IDESC_O, true);
          }
        }
        if (!ok) break;
        tc::commit_lane0(smem_addr(bars + kPvDone + t));
        if (t == kTcTiles - 1) tc::commit_lane0(smem_addr(bars + kVEmpty + sv));  // both P V of stage j issued
        if (j + 1 < nkv) {
          if (t == 0) ok = mbar_wait(bars + kKFull + (j + 1) % kTcKStages, ((j + 1) / kTcKStages) & 1, p.err);
          // S_t is rewritten only after the P_t V that reads it has completed
          if (ok) ok = mbar_wait(bars + kPvDone + t, j & 1, p.err);
          ok = __all_sync(kFullMask, ok);
          if (ok) {
            tc::fence_after_sync();
            issue_qk(t, j + 1);
          }
        }
      }
    }
    // every MMA of this warp done before TMEM is freed, whatever happened above
    tc::commit_lane0(smem_addr(bars + kDrain));
    mbar_wait(bars + kDrain, 0, p.err);
  } else {
    // ---------------------------------------------------------- softmax rows
    const int t = warp / 4;                        // this warpgroup's tile
    const int r = threadIdx.x - 128 * t;           // this thread's row (TMEM lane)
    const int tok = t * QT + r / G, head = g * G + r % G;
    const bool ok = i0 + tok < n;
    const int lim = ok ? pos0 + tok : p_max;       // causal limit of the row
    const uint32_t trow = tmem + (static_cast<uint32_t>((warp % 4) * 32) << 16);
    const uint32_t scol = kColS + kTcRows * t, ocol = kColO + kTcRows * t;
    const float scale = p.qk_scale_log2;
    float m_used = -INFINITY, l = 0.f;             // max the weights are taken against; row sum
    for (int j = 0; j < nkv; ++j) {
      mbar_wait(bars + kSFull + t, j & 1, p.err);
      tc::fence_after_sync();
      const int t0 = (st0 + j) * kTcKv;            // position of the stage's first token
      // Stages that reach past a row's position take the masked path, for
      // the whole warp (one path per warp, not one per row)
      const bool masked = __any_sync(kFullMask, t0 + kTcKv - 1 > lim);
      // pass 1: the row's maximum over the stage (four loads, one wait)
      float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
      {
        uint32_t v[kTcKv];
#pragma unroll
        for (int h = 0; h < kTcKv / 32; ++h)
          tc::ld_32x32b_x32(trow + scol + 32 * h, *reinterpret_cast<uint32_t(*)[32]>(v + 32 * h));
        tc::wait_ld();
        if (!masked) {
          // four independent chains of three-input maxima
#pragma unroll
          for (int c = 0; c < kTcKv; c += 8) {
            mx0 = fmax3(mx0, __uint_as_float(v[c]), __uint_as_float(v[c + 1]));
            mx1 = fmax3(mx1, __uint_as_float(v[c + 2]), __uint_as_float(v[c + 3]));
            mx2 = fmax3(mx2, __uint_as_float(v[c + 4]), __uint_as_float(v[c + 5]));
            mx3 = fmax3(mx3, __uint_as_float(v[c + 6]), __uint_as_float(v[c + 7]));
          }
        } else {
#pragma unroll
          for (int c = 0; c < kTcKv; c += 2) {
            mx0 = fmaxf(mx0, t0 + c <= lim ? __uint_as_float(v[c]) : -INFINITY);
            mx1 = fmaxf(mx1, t0 + c + 1 <= lim ? __uint_as_float(v[c + 1]) : -INFINITY);
          }
        }
      }
      const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
      // every row sees token 0 in the first stage, so m_new is finite
      const float m_new = fmaxf(m_used, mx * scale);
      const bool need = m_new > m_used + kRescaleSlack;
      const float alpha = fast_exp2(m_used - m_new);  // 0 on the first stage (m_used = -inf)
      if (need) {
        l *= alpha;
        m_used = m_new;
      }
      if (j >= 1 && __any_sync(kFullMask, need)) {
        // rescale O_t: idle now, since P_t V of stage j-1 completed before
        // S_t(j) was written
        const float f = need ? alpha : 1.f;
#pragma unroll
        for (int c4 = 0; c4 < D / 32; ++c4) {
          uint32_t v[32];
          tc::ld_32x32b_x32(trow + ocol + 32 * c4, v);
          tc::wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * f);
          tc::st_32x32b_x32(trow + ocol + 32 * c4, v);
        }
      }
      if (j == nkv - 1) {
        // V rows from z0 on may hold anything: past the sequence, or not
        // loaded.  Once the stage's copies have landed (a copy that landed
        // later would overwrite the zeros with the block's tail), both
        // warpgroups zero them (the same values), each before the first
        // half of its own P_t V may read the stage.
        const int loaded = min(kTcKv / kBlockSize, (p_max - t0) / kBlockSize + 1) * kBlockSize;
        const int z0 = min(L - t0, loaded);
        if (z0 < kTcKv) {
          mbar_wait(bars + kVFull + j % kTcVStages, (j / kTcVStages) & 1, p.err);
          unsigned char* vst = sm + lay.v + (j % kTcVStages) * STAGE;
          for (int idx = r; idx < (kTcKv - z0) * BOXES * 8; idx += kTcRows) {
            const int vr = z0 + idx / (BOXES * 8), rest = idx % (BOXES * 8);
            *reinterpret_cast<uint4*>(vst + (rest >> 3) * kTcKv * 128 + vr * 128 + (rest & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
      fence_proxy_async_smem();  // zeroed V rows visible to the tensor cores
      // pass 2: P = 2^(scale s - m_used) <= 2^8, 32 tokens (one chunk of S_t's
      // columns) at a time, two per packed fp32 operation.  Chunk h's weights
      // go over its own 32 columns, which it has just read: bf16 high parts in
      // [32h, 32h + 16), low parts in [32h + 16, 32h + 32), two per column.
      const float2 sc2 = make_float2(scale, scale), nm2 = make_float2(-m_used, -m_used);
      float2 l2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};  // two independent sum chains
      uint32_t v[64];
      tc::ld_32x32b_x32(trow + scol, *reinterpret_cast<uint32_t(*)[32]>(v));
      tc::ld_32x32b_x32(trow + scol + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
      tc::wait_ld();
#pragma unroll 1
      for (int h2 = 0; h2 < kTcKv / 64; ++h2) {  // two chunks of 32 per TMEM read
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int h = 2 * h2 + hh;
          uint32_t hi[16], lo[16];
          if (!masked) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float2 y = ffma2(make_float2(__uint_as_float(v[32 * hh + 2 * e]), __uint_as_float(v[32 * hh + 2 * e + 1])),
                                     sc2, nm2);
              const float2 w = make_float2(fast_exp2(y.x), fast_exp2(y.y));
              l2[e & 1] = fadd2(l2[e & 1], w);
              split_bf16x2(w.x, w.y, hi[e], lo[e]);
            }
          } else {
            const int tb = t0 + 32 * h;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float x0 = tb + 2 * e <= lim ? __uint_as_float(v[32 * hh + 2 * e]) : -INFINITY;
              const float x1 = tb + 2 * e + 1 <= lim ? __uint_as_float(v[32 * hh + 2 * e + 1]) : -INFINITY;
              const float2 y = ffma2(make_float2(x0, x1), sc2, nm2);
              const float2 w = make_float2(fast_exp2(y.x), fast_exp2(y.y));
              l2[e & 1] = fadd2(l2[e & 1], w);
              split_bf16x2(w.x, w.y, hi[e], lo[e]);
            }
          }
          tc::st_32x32b_x16(trow + scol + 32 * h, hi);
          tc::st_32x32b_x16(trow + scol + 32 * h + 16, lo);
        }
        if (h2 == 0) {  // the first 64 tokens' weights: their half of P_t V may start
          // the next 64 scores are read while these weights land in TMEM
          tc::ld_32x32b_x32(trow + scol + 64, *reinterpret_cast<uint32_t(*)[32]>(v));
          tc::ld_32x32b_x32(trow + scol + 96, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
          // V_j landed before the stage's first arrival (the MMA warp relies on it)
          if (t == 0) mbar_wait(bars + kVFull + j % kTcVStages, (j / kTcVStages) & 1, p.err);
          tc::wait_st();
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(bars + kPHalf + t);
          tc::wait_ld();
        }
      }
      l += (l2[0].x + l2[1].x) + (l2[0].y + l2[1].y);
      tc::wait_st();
      tc::fence_before_sync();  // P stores in TMEM before the arrival
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + kPFull + t);
    }

    // ---- O / l for this row, after the last P V
    mbar_wait(bars + kPvDone + t, (nkv - 1) & 1, p.err);
    tc::fence_after_sync();
    OutT* dst = reinterpret_cast<OutT*>(p.out) + static_cast<int64_t>(q0 + i0 + tok) * p.o_st +
                static_cast<int64_t>(head) * p.o_sh;
    if (nch == 1) {
      const float inv = 1.f / l;
#pragma unroll
      for (int c4 = 0; c4 < D / 32; ++c4) {
        uint32_t v[32];
        tc::ld_32x32b_x32(trow + ocol + 32 * c4, v);
        tc::wait_ld();
        if (ok) store_row32(dst + 32 * c4, v, inv);
      }
    } else {
      // This chunk's partial row: O (against m_used, not divided), m_used
      // and l.  Partial rows of (item, KV head g) sit at
      // ((item Hkv + g) max_chunks + chunk) rows + row.
      const int64_t base = (static_cast<int64_t>(item) * p.Hkv + g) * chunk_slots;
      const int row = t * kTcRows + r;
      constexpr int kRows = kTcTiles * kTcRows;
      float* po = p.ws_o + ((base + ch) * kRows + row) * D;
#pragma unroll
      for (int c4 = 0; c4 < D / 32; ++c4) {
        uint32_t v[32];
        tc::ld_32x32b_x32(trow + ocol + 32 * c4, v);
        tc::wait_ld();
#pragma unroll
        for (int c = 0; c < 32; c += 4)
          *reinterpret_cast<uint4*>(po + 32 * c4 + c) = make_uint4(v[c], v[c + 1], v[c + 2], v[c + 3]);
      }
      *reinterpret_cast<float2*>(p.ws_ml + ((base + ch) * kRows + row) * 2) = make_float2(m_used, l);
      // Arrival, as in the decode's split merge: the barrier orders every
      // softmax thread's partial stores before thread 0's acquire-release
      // atomic, whose release half publishes them; in the last chunk to
      // arrive its acquire half and the barrier order the other chunks'
      // partials before every thread's reads.
      int* counter = p.counters + static_cast<int64_t>(item) * p.Hkv + g;
      volatile int* last_flag = reinterpret_cast<volatile int*>(bars + kSlot) + 1;
      named_barrier(1, kTcSoftmaxWarps * 32);
      if (threadIdx.x == 0) {
        int old;
        asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
        *last_flag = old == nch - 1 ? 1 : 0;
      }
      named_barrier(1, kTcSoftmaxWarps * 32);
      if (*last_flag) {
        // merge the row's nch partials: M = max_c m_c, w_c = 2^(m_c - M),
        // out = sum_c w_c O_c / sum_c w_c l_c (every chunk saw a token of
        // the row, so every l_c > 0 and m_c is finite)
        float M = -INFINITY;
        for (int c = 0; c < nch; ++c) M = fmaxf(M, __ldcg(p.ws_ml + ((base + c) * kRows + row) * 2));
        float den = 0.f;
        for (int c = 0; c < nch; ++c) {
          const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.ws_ml + ((base + c) * kRows + row) * 2));
          den = fmaf(fast_exp2(ml.x - M), ml.y, den);
        }
        const float inv = 1.f / den;
#pragma unroll
        for (int c4 = 0; c4 < D / 32; ++c4) {
          float acc[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) acc[e] = 0.f;
          for (int c = 0; c < nch; ++c) {
            const float w = fast_exp2(__ldcg(p.ws_ml + ((base + c) * kRows + row) * 2) - M);
            const float4* src = reinterpret_cast<const float4*>(p.ws_o + ((base + c) * kRows + row) * D + 32 * c4);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float4 x = __ldcg(src + e);
              acc[4 * e] = fmaf(w, x.x, acc[4 * e]);
              acc[4 * e + 1] = fmaf(w, x.y, acc[4 * e + 1]);
              acc[4 * e + 2] = fmaf(w, x.z, acc[4 * e + 2]);
              acc[4 * e + 3] = fmaf(w, x.w, acc[4 * e + 3]);
            }
          }
          uint32_t v[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(acc[e]);
          if (ok) store_row32(dst + 32 * c4, v, inv);
        }
        if (threadIdx.x == 0) *counter = 0;  // ready for the next call
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == kTcMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, int G, typename OutT>
cudaError_t launch_tc_typed(const PrefillParams& p, const CUtensorMap& tmq, const CUtensorMap& tmk,
                            const CUtensorMap& tmv, cudaStream_t stream) {
  auto kernel = paged_prefill_tc_kernel<D, G, OutT>;
  static std::atomic<int> smem_set[64];  // one record per instantiation
  const int smem = tc_layout(D).total;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) dev = 63;
  if (!smem_set[dev].load(std::memory_order_relaxed)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    smem_set[dev].store(1);
  }
  const int64_t items = prefill_tc_items(p.T, p.B, G);  // >= sum of ceil(n_b / QT2)
  const int64_t ctas = items * std::max(1, p.max_chunks) * p.Hkv;
  if (ctas > 0x7fffffff) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(ctas));
  kernel<<<grid, kTcThreads, smem, stream>>>(tmq, tmk, tmv, p);
  return cudaGetLastError();
}

template <int D, typename OutT>
cudaError_t launch_tc_g(const PrefillParams& p, const CUtensorMap& tmq, const CUtensorMap& tmk,
                        const CUtensorMap& tmv, int G, cudaStream_t stream) {
  switch (G) {
    case 1: return launch_tc_typed<D, 1, OutT>(p, tmq, tmk, tmv, stream);
    case 2: return launch_tc_typed<D, 2, OutT>(p, tmq, tmk, tmv, stream);
    case 4: return launch_tc_typed<D, 4, OutT>(p, tmq, tmk, tmv, stream);
    case 8: return launch_tc_typed<D, 8, OutT>(p, tmq, tmk, tmv, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int64_t prefill_tc_items(int64_t T, int64_t B, int G) {
  const int64_t qt2 = kTcTiles * (kTcRows / G);  // query tokens per work item
  return (T + qt2 - 1) / qt2 + B;
}

cudaError_t launch_prefill_tc(const PrefillParams& p, const CUtensorMap& tmq, const CUtensorMap& tmk,
                              const CUtensorMap& tmv, int D, int G, bool out_bf16, cudaStream_t stream) {
  if (p.B == 0 || p.T == 0) return cudaSuccess;
  if (D == 128) {
    return out_bf16 ? launch_tc_g<128, __nv_bfloat16>(p, tmq, tmk, tmv, G, stream)
                    : launch_tc_g<128, float>(p, tmq, tmk, tmv, G, stream);
  }
  if (D == 64) {
    return out_bf16 ? launch_tc_g<64, __nv_bfloat16>(p, tmq, tmk, tmv, G, stream)
                    : launch_tc_g<64, float>(p, tmq, tmk, tmv, G, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace forge
