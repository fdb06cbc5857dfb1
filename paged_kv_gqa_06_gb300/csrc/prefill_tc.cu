// Paged prefill on the 5th-generation tensor cores (tcgen05.mma, TMEM).
//
// What it computes is the prefill of prefill.cu ("Make the Engine Talk",
// 1.2: one forward pass over all of a prompt's tokens, which fills the KV
// cache): query token i of sequence b's run of n_b tokens sits at position
// p = L_b - n_b + i and attends to every cached position t <= p of its KV
// head's group.
//
// One CTA per (query tile, KV head g); a query tile is M = 128 MMA rows:
// 128 / G consecutive query tokens x the G heads of group g (row r is token
// r / G, head g*G + r % G).  Six warps with fixed roles:
//   * warp 4 (producer) loads the Q tile once (a 3-D TMA box of 64 dims x G
//     heads x 128/G tokens, which lands as 128 K-major rows) and streams the
//     sequence's K and V, 64 tokens (4 blocks) per stage, through the block
//     table into a 3-stage ring, up to the tile's last query position.  The
//     third stage is the Q tile's own space, filled once Q is in TMEM;
//   * warps 0-3 (softmax) own one row each (warp w reads TMEM lanes
//     32w..32w+31).  First each thread copies its row of Q from shared memory
//     into TMEM, where it is the A operand of every QK^T.  Per tile: load the
//     row of S, mask by position (only on tiles that reach past the row's
//     position), and keep a running maximum that only moves when the row's
//     maximum grows by more than 8 in log2 units, so the weights stay <= 2^8
//     and O in TMEM is rescaled rarely.  The weights P = 2^(scale s - m) are
//     stored over the row's S in TMEM, two per column in its first 32
//     columns, as bf16 high and low parts (low in the next 32 columns; two
//     MMAs keep ~16 bits of each weight, as in the decode).  A weight rounded
//     to bf16 once would lose up to 2^-8 of itself, which at |V| near 8 is as
//     large as a bf16 output's own rounding.  At the end O is divided by the
//     row sum and stored;
//   * warp 5 (MMA) owns 256 TMEM columns: S (64), Q (D / 2: two bf16 per
//     column) and the output accumulator O (D).  Its lane 0 issues
//     S_j = Q K_j^T (M 128, N 64, K = D; Q from TMEM, K K-major straight from
//     the TMA layout) and O += P_j V_j (M 128, N = D, K 64; P from TMEM over
//     S, V MN-major as it lies in the stage), each as soon as its inputs are
//     ready: S_{j+1} overwrites S, so it waits for P_j V_j.  tcgen05.commit on
//     mbarriers tracks completion and frees stages.  With Q in TMEM, QK^T
//     reads only K from shared memory: on this GPU an MMA with both operands
//     in shared memory runs at well under the rate of one with A in TMEM.
// Shared memory is 98 KB and TMEM 256 columns per CTA, so two CTAs share an
// SM: while one CTA's softmax runs, the other's MMAs keep the tensor cores
// busy.
// V rows that may hold anything (the tail of the last block, or blocks the
// last stage did not load) are zeroed before P V reads them: P is 0 there,
// but 0 * NaN is NaN.  Every mbarrier wait is bounded; the MMA warp drains
// its own MMAs before TMEM is freed.
#include <atomic>

#include "common.cuh"
#include "tcgen05.cuh"

namespace forge {
namespace {

constexpr int kTcRows = 128;                 // MMA M
constexpr int kTcKv = 64;                    // tokens per stage (MMA N of S, K of P V)
constexpr int kTcStages = 3;                 // K/V ring depth: 2 stages + the Q tile's space once Q is in TMEM
constexpr int kTcThreads = 6 * 32;
constexpr int kSoftmaxThreads = 128;
constexpr int kTmemCols = 256;
constexpr int kColS = 0;                     // S (and P over it): 64 columns
constexpr int kColQ = 64;                    // Q, the A operand of QK^T: D / 2 columns (2 bf16 each)
constexpr int kColO = 128;                   // O: D columns
constexpr float kRescaleSlack = 8.0f;        // log2 units: weights stay <= 2^8
constexpr unsigned kFullMask = 0xffffffffu;

struct TcLayout {
  int q, kv, bars, total;
};

// Q [BOXES][128 rows][128 B] | 2 x ([K: BOXES][64][128 B], [V: same]) |
// mbarriers, TMEM slot.  Offsets from a 1024-byte-aligned base.  The third
// K/V stage uses Q's space once Q has been copied into TMEM.
__host__ __device__ constexpr TcLayout tc_layout(int D) {
  const int boxes = D / 64;
  TcLayout l{};
  l.q = 0;
  l.kv = l.q + boxes * kTcRows * 128;
  l.bars = l.kv + 2 * 2 * boxes * kTcKv * 128;  // stages 0 and 1; stage 2 reuses Q's space
  l.total = l.bars + 16 * 8 + 1024;          // barriers + slot, + alignment slack
  return l;
}

// Shared-memory offset of K/V stage st: two stages after Q, the third in
// Q's own space (free once Q has been copied into TMEM; same size as a stage).
__host__ __device__ constexpr int stage_offset(const TcLayout& l, int st, int stage_bytes) {
  return st < 2 ? l.kv + st * stage_bytes : l.q;
}

// mbarrier slots
constexpr int kQFull = 0;
constexpr int kKvFull = 1;                   // [kTcStages]
constexpr int kKvEmpty = kKvFull + kTcStages;
constexpr int kSFull = kKvEmpty + kTcStages; // S_j written
constexpr int kPFull = kSFull + 1;           // P_j written over S_j (one arrival per softmax warp)
constexpr int kPvDone = kPFull + 1;          // P_j V_j done: S free for S_{j+1}
constexpr int kDrain = kPvDone + 1;
constexpr int kQTmem = kDrain + 1;           // Q copied into TMEM (one arrival per softmax warp)
constexpr int kSlot = kQTmem + 1;            // TMEM address (4 bytes) after the barriers

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

// Find (sequence, first query token) of tile `tile_id` from query_start: a
// warp scan over the sequences' tile counts, the same answer in every warp.
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

template <int D, int G, typename OutT>
__global__ void __launch_bounds__(kTcThreads, 2)
    paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                            const __grid_constant__ CUtensorMap tmv, const PrefillParams p) {
  constexpr int QT = kTcRows / G;            // query tokens per CTA
  constexpr int BOXES = D / 64;
  constexpr int KSTEPS = D / 16;
  constexpr TcLayout lay = tc_layout(D);
  constexpr int KV_HALF = BOXES * kTcKv * 128;   // K (or V) part of a stage
  constexpr uint32_t IDESC_S = tc::idesc_bf16_f32(kTcRows, kTcKv, false);
  constexpr uint32_t IDESC_O = tc::idesc_bf16_f32(kTcRows, D, true);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.y;
  const int tile_id = static_cast<int>(gridDim.x - 1 - blockIdx.x);  // later (longer) tiles first

  // query_start must start at 0, never decrease and end within the T rows
  if (blockIdx.x == 0 && g == 0 && warp == 0) {
    bool bad = lane == 0 && __ldg(p.query_start) != 0;
    for (int b = lane; b < p.B; b += 32) {
      const int s0 = __ldg(p.query_start + b), s1 = __ldg(p.query_start + b + 1);
      bad |= s1 < s0 || s1 > p.T;
    }
    if (__any_sync(kFullMask, bad) && lane == 0) record_error(p.err, kDevErrQuery);
  }

  int b, i0;
  find_tile<QT>(p, tile_id, lane, b, i0);
  if (b < 0) return;  // past the last tile

  const int q0 = __ldg(p.query_start + b);
  const int n = __ldg(p.query_start + b + 1) - q0;
  const int L = __ldg(p.context_lens + b);
  if (L < 0 || L > p.MB * kBlockSize || n > L || q0 < 0 || q0 + n > p.T) {
    if (threadIdx.x == 0) record_error(p.err, (L < 0 || L > p.MB * kBlockSize) ? kDevErrLength : kDevErrQuery);
    return;
  }
  const int pos0 = L - n + i0;                     // position of the tile's first query token
  const int p_max = pos0 + min(QT, n - i0) - 1;    // of its last (<= L - 1)
  const int nkv = p_max / kTcKv + 1;               // stages up to and including p_max

  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                       ~static_cast<uintptr_t>(1023));
  const uint32_t sm_s = smem_addr(sm);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + lay.bars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kSlot);

  if (threadIdx.x == 0) {
    mbar_init(bars + kQFull, 1);
    for (int i = 0; i < kTcStages; ++i) {
      mbar_init(bars + kKvFull + i, 1);
      mbar_init(bars + kKvEmpty + i, 1);
    }
    mbar_init(bars + kSFull, 1);
    mbar_init(bars + kPFull, 4);   // one arrival per softmax warp
    mbar_init(bars + kPvDone, 1);
    mbar_init(bars + kDrain, 1);
    mbar_init(bars + kQTmem, 4);
    fence_barrier_init();
  }
  if (warp == 5) {
    tc::tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(bars + kQFull, BOXES * kTcRows * 128);
#pragma unroll
      for (int c = 0; c < BOXES; ++c)
        tma_load_3d(sm + lay.q + c * kTcRows * 128, &tmq, c * 64, g * G, q0 + i0, bars + kQFull);
      const int32_t* row = p.block_tables + static_cast<int64_t>(b) * p.bt_sb;
      for (int j = 0; j < nkv; ++j) {
        const int st = j % kTcStages, use = j / kTcStages;
        if (use > 0)
          mbar_wait(bars + kKvEmpty + st, (use - 1) & 1, p.err);  // stage released by P V
        else if (st == 2)
          mbar_wait(bars + kQTmem, 0, p.err);  // Q's space: free once Q is in TMEM
        unsigned char* kst = sm + stage_offset(lay, st, 2 * KV_HALF);
        int pb[4];
        uint32_t bytes = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int jb = 4 * j + u;
          pb[u] = -1;
          if (jb * kBlockSize <= p_max) {
            const int e = __ldg(row + jb);
            if (static_cast<unsigned>(e) < static_cast<unsigned>(p.NB)) {
              pb[u] = e;
              bytes += 2 * BOXES * kBlockSize * 128;
            } else {
              record_error(p.err, kDevErrBlockId);
            }
          }
        }
        if (bytes) {
          mbar_arrive_expect_tx(bars + kKvFull + st, bytes);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            if (pb[u] < 0) continue;
#pragma unroll
            for (int c = 0; c < BOXES; ++c) {
              const int off = c * kTcKv * 128 + u * kBlockSize * 128;
              tma_load_4d(kst + off, &tmk, c * 64, 0, g, pb[u], bars + kKvFull + st);
              tma_load_4d(kst + KV_HALF + off, &tmv, c * 64, 0, g, pb[u], bars + kKvFull + st);
            }
          }
        } else {
          mbar_arrive(bars + kKvFull + st);  // nothing to copy (a bad id is recorded above)
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issue
    // Issue each MMA group as soon as its inputs are ready, whichever comes
    // first: S_j = Q K_j^T needs stage j loaded and S buffer j % 2 free
    // (P_{j-2} V done); O += P_j V_j needs P_j written.  Waiting for one
    // would hold back the other and stall the ring.
    if (lane == 0) {
      mbar_wait(bars + kQTmem, 0, p.err);
      tc::fence_after_sync();
      int next_qk = 0, next_pv = 0;
      uint64_t last = global_timer_ns();
      while (next_pv < nkv) {
        bool progressed = false;
        if (next_qk < nkv && next_qk == next_pv) {  // one S buffer: P_{j-1} V_{j-1} issued first
          const int j = next_qk, st = j % kTcStages;
          if (mbar_try_wait(bars + kKvFull + st, (j / kTcStages) & 1) &&
              (j < 1 || mbar_try_wait(bars + kPvDone, (j - 1) & 1))) {
            tc::fence_after_sync();
            const uint32_t kst = sm_s + stage_offset(lay, st, 2 * KV_HALF);
#pragma unroll
            for (int k = 0; k < KSTEPS; ++k) {
              const uint64_t bd = tc::smem_desc_sw128(kst + (k >> 2) * kTcKv * 128 + (k & 3) * 32, 0, 1024);
              tc::mma_bf16_ts(tmem + kColS, tmem + kColQ + 8 * k, bd, IDESC_S, k > 0);
            }
            tc::commit(smem_addr(bars + kSFull));
            ++next_qk;
            progressed = true;
          }
        }
        if (next_pv < next_qk) {
          const int jp = next_pv, stp = jp % kTcStages;
          if (mbar_try_wait(bars + kPFull, jp & 1)) {
            tc::fence_after_sync();
            const uint32_t vst = sm_s + stage_offset(lay, stp, 2 * KV_HALF) + KV_HALF;
            const uint32_t phi = tmem + kColS, plo = phi + kTcKv / 2;  // P over S in TMEM
#pragma unroll
            for (int kk = 0; kk < kTcKv / 16; ++kk) {
              const uint64_t bd = tc::smem_desc_sw128(vst + kk * 16 * 128, kTcKv * 128, 1024);
              tc::mma_bf16_ts(tmem + kColO, phi + 8 * kk, bd, IDESC_O, jp > 0 || kk > 0);
              tc::mma_bf16_ts(tmem + kColO, plo + 8 * kk, bd, IDESC_O, true);
            }
            tc::commit(smem_addr(bars + kPvDone));
            tc::commit(smem_addr(bars + kKvEmpty + stp));
            ++next_pv;
            progressed = true;
          }
        }
        if (progressed) {
          last = global_timer_ns();
        } else if (global_timer_ns() - last > kWaitLimitNs) {
          record_error(p.err, kDevErrTimeout);
          break;
        }
      }
      // every MMA of this thread done before TMEM is freed, whatever happened above
      tc::commit(smem_addr(bars + kDrain));
      mbar_wait(bars + kDrain, 0, p.err);
    }
  } else {
    // ---------------------------------------------------------- softmax rows
    const int r = threadIdx.x;                     // this thread's row (TMEM lane)
    const int tok = r / G, head = g * G + r % G;
    const bool ok = i0 + tok < n;
    const int lim = ok ? pos0 + tok : p_max;       // causal limit of the row
    const uint32_t trow = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const float scale = p.qk_scale_log2;
    // This row of Q into TMEM (the A operand of QK^T): from the TMA tile in
    // shared memory (128-byte rows, 16-byte chunks swizzled by row % 8), 32
    // columns of two bf16 per box of 64 dims
    mbar_wait(bars + kQFull, 0, p.err);
#pragma unroll
    for (int c = 0; c < BOXES; ++c) {
      uint32_t v[32];
      const unsigned char* qrow = sm + lay.q + c * kTcRows * 128 + r * 128;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        const uint4 w = *reinterpret_cast<const uint4*>(qrow + ((ch ^ (r & 7)) * 16));
        v[4 * ch] = w.x;
        v[4 * ch + 1] = w.y;
        v[4 * ch + 2] = w.z;
        v[4 * ch + 3] = w.w;
      }
      tc::st_32x32b_x32(trow + kColQ + 32 * c, v);
    }
    tc::wait_st();
    tc::fence_before_sync();
    fence_proxy_async_smem();  // the Q reads above before the TMA engine refills this space
    __syncwarp();
    if (lane == 0) mbar_arrive(bars + kQTmem);
    float m_used = -INFINITY, l = 0.f;             // max the weights are taken against; row sum
    for (int j = 0; j < nkv; ++j) {
      mbar_wait(bars + kSFull, j & 1, p.err);
      tc::fence_after_sync();
      float s[kTcKv];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t v[32];
        tc::ld_32x32b_x32(trow + kColS + 32 * h, v);
        tc::wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) s[32 * h + c] = __uint_as_float(v[c]);
      }

      const int t0 = j * kTcKv;
      if (t0 + kTcKv - 1 > lim) {  // the tile reaches past this row's position
#pragma unroll
        for (int c = 0; c < kTcKv; ++c) s[c] = t0 + c <= lim ? s[c] : -INFINITY;
      }
      // the row's maximum as a tree (6 levels, not a chain of 64)
      float mt[kTcKv / 2];
#pragma unroll
      for (int c = 0; c < kTcKv / 2; ++c) mt[c] = fmaxf(s[c], s[c + kTcKv / 2]);
#pragma unroll
      for (int w = kTcKv / 4; w >= 1; w >>= 1) {
#pragma unroll
        for (int c = 0; c < w; ++c) mt[c] = fmaxf(mt[c], mt[c + w]);
      }
      const float mx = mt[0];
      // every row sees token 0 in the first stage, so m_new is finite
      const float m_new = fmaxf(m_used, mx * scale);
      const bool need = m_new > m_used + kRescaleSlack;
      const float alpha = fast_exp2(m_used - m_new);  // 0 on the first stage (m_used = -inf)
      if (need) {
        l *= alpha;
        m_used = m_new;
      }
      if (j >= 1 && __any_sync(kFullMask, need)) {
        // rescale O: every P V so far (the last is tile j-1) must be finished
        mbar_wait(bars + kPvDone, (j - 1) & 1, p.err);
        tc::fence_after_sync();
        const float f = need ? alpha : 1.f;
#pragma unroll
        for (int c4 = 0; c4 < D / 32; ++c4) {
          uint32_t v[32];
          tc::ld_32x32b_x32(trow + kColO + 32 * c4, v);
          tc::wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * f);
          tc::st_32x32b_x32(trow + kColO + 32 * c4, v);
        }
        tc::wait_st();
      }
      // P = 2^(scale s - m_used) <= 2^8 over S in TMEM, two weights per
      // column in columns [0, 32) of the buffer as bf16 high parts and the
      // low parts in [32, 64); in two halves of 32 weights
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float a = fast_exp2(fmaf(s[32 * h + 2 * e], scale, -m_used));
          const float c = fast_exp2(fmaf(s[32 * h + 2 * e + 1], scale, -m_used));
          l += a + c;
          split_bf16x2(a, c, hi[e], lo[e]);
        }
        tc::st_32x32b_x16(trow + kColS + 16 * h, hi);
        tc::st_32x32b_x16(trow + kColS + kTcKv / 2 + 16 * h, lo);
      }
      tc::wait_st();
      if (j == nkv - 1) {
        // V rows from z0 on may hold anything: past the sequence, or not loaded
        const int loaded = min(kTcKv / kBlockSize, (p_max - t0) / kBlockSize + 1) * kBlockSize;
        const int z0 = min(L - t0, loaded);
        if (z0 < kTcKv) {
          unsigned char* vst = sm + stage_offset(lay, j % kTcStages, 2 * KV_HALF) + KV_HALF;
          for (int idx = r; idx < (kTcKv - z0) * BOXES * 8; idx += kSoftmaxThreads) {
            const int vr = z0 + idx / (BOXES * 8), rest = idx % (BOXES * 8);
            *reinterpret_cast<uint4*>(vst + (rest >> 3) * kTcKv * 128 + vr * 128 + (rest & 7) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
        }
      }
      fence_proxy_async_smem();  // zeroed V rows visible to the tensor cores
      tc::fence_before_sync();   // P stores in TMEM before the arrival
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + kPFull);
    }

    // ---- O / l for this row, after the last P V
    mbar_wait(bars + kPvDone, (nkv - 1) & 1, p.err);
    tc::fence_after_sync();
    const float inv = 1.f / l;
    OutT* dst = reinterpret_cast<OutT*>(p.out) + static_cast<int64_t>(q0 + i0 + tok) * p.o_st +
                static_cast<int64_t>(head) * p.o_sh;
#pragma unroll
    for (int c4 = 0; c4 < D / 32; ++c4) {
      uint32_t v[32];
      tc::ld_32x32b_x32(trow + kColO + 32 * c4, v);
      tc::wait_ld();
      if (ok) store_row32(dst + 32 * c4, v, inv);
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 5) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, int G, typename OutT>
cudaError_t launch_tc_typed(const PrefillParams& p, const CUtensorMap& tmq, const CUtensorMap& tmk,
                            const CUtensorMap& tmv, cudaStream_t stream) {
  constexpr int QT = kTcRows / G;
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
  const int64_t tiles = (static_cast<int64_t>(p.T) + QT - 1) / QT + p.B;  // >= sum of ceil(n_b / QT)
  if (tiles > 0x7fffffff) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(p.Hkv));
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
