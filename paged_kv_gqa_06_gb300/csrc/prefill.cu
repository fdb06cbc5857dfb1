// Paged prefill: causal attention of a run of new query tokens per sequence
// over that sequence's paged KV cache.
//
// "Make the Engine Talk", 1.2: the prefill runs one forward pass over all of
// a prompt's tokens at once and fills the KV cache; forge-engine README,
// "What it implements": prefill and decode are separate engine paths over the
// same paged cache.  With the run's K/V already appended, query token i of
// sequence b (n_b query tokens, L_b cached tokens) sits at position
// p = L_b - n_b + i, and for query head h (G = Hq / Hkv):
//   out[i, h, :] = sum_{t <= p} softmax_t(scale * q[i, h, :] . K[t, h/G, :]) V[t, h/G, :]
// The decode is the n_b = 1 case.
//
// Work decomposition.  Unlike the decode this is a dense contraction: every
// K/V byte meets 64/G query tokens of the G heads of its group, so it runs on
// the tensor cores with K/V read from shared memory many times.
//   * One CTA per (query tile, KV head g).  A query tile is 64 MMA rows:
//     64/G consecutive query tokens x the G heads of group g (row r is token
//     r / G, head g*G + r % G).  Tiles are numbered across the batch in
//     query_start order and found on the device by a warp scan, so nothing
//     is read back to the host.  Later tiles of a sequence attend to more
//     tokens; the grid runs them first.
//   * Warp 4 is the producer: it streams the sequence's K/V through the block
//     table, 32 tokens (two blocks) per stage, into a ring of stages with
//     tiled TMA copies (the same tensor maps and 128-byte swizzle as the
//     decode), and only up to the tile's last query position.
//   * Warps 0-3 each own 16 rows.  Per stage: S = Q K^T on mma.sync
//     m16n8k16 (Q fragments in registers, K from the swizzled tile by
//     ldmatrix), the causal mask by position, an online softmax in log2 units
//     (running max and sum per row, rescaling the accumulator), then
//     O += P V with P split into bf16 high and low parts (two MMAs), so the
//     weights keep ~16 bits, and V read with transposing ldmatrix.
//   * V rows that may hold anything (the tail of the sequence's last block,
//     or a block the last stage did not load) are zeroed before P V: their P
//     is 0, but 0 * NaN is NaN.
#include <atomic>

#include "common.cuh"

namespace forge {
namespace {

constexpr int kPfWarps = 4;                      // consumer warps, 16 MMA rows each
constexpr int kPfRows = kPfWarps * 16;           // query rows (tokens x heads) per CTA
constexpr int kPfConsumers = kPfWarps * 32;
constexpr int kPfThreads = kPfConsumers + 32;    // + one producer warp
constexpr int kKvTokens = 2 * kBlockSize;        // tokens per pipeline stage
constexpr int kPfStages = 3;
constexpr unsigned kFull = 0xffffffffu;

__host__ __device__ constexpr int tile_bytes(int D) { return kBlockSize * D * 2; }

// ring of kPfStages stages [K block 0 | K block 1 | V block 0 | V block 1]
// (1024-byte aligned for the swizzle) | full / empty mbarriers
__host__ __device__ constexpr size_t prefill_smem_bytes(int D) {
  return 1024 + static_cast<size_t>(kPfStages) * 4 * tile_bytes(D) + 2 * kPfStages * 8;
}

__device__ __forceinline__ uint32_t ldg_u32(const __nv_bfloat16* p) {
  return __ldg(reinterpret_cast<const uint32_t*>(p));
}

__device__ __forceinline__ void store2(float* p, float x, float y) {
  *reinterpret_cast<float2*>(p) = make_float2(x, y);
}
__device__ __forceinline__ void store2(__nv_bfloat16* p, float x, float y) {
  *reinterpret_cast<uint32_t*>(p) = pack_bf16x2(x, y);
}

template <int D, int G, typename OutT>
__global__ void __launch_bounds__(kPfThreads) paged_prefill_kernel(const __grid_constant__ CUtensorMap tmk,
                                                                   const __grid_constant__ CUtensorMap tmv,
                                                                   const PrefillParams p) {
  constexpr int QT = kPfRows / G;  // query tokens per CTA
  constexpr int KSTEPS = D / 16;
  constexpr int BOXES = D / kBoxDims;
  constexpr int TILE = tile_bytes(D);
  constexpr int STAGE = 4 * TILE;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // One-dimensional grid, the KV head fastest, later (longer) tiles first:
  // the order holds across the heads too (CTAs are dispatched by index).
  const int g = static_cast<int>(blockIdx.x % static_cast<unsigned>(p.Hkv));
  const int tile_id = static_cast<int>(gridDim.x / static_cast<unsigned>(p.Hkv)) - 1 -
                      static_cast<int>(blockIdx.x / static_cast<unsigned>(p.Hkv));

  // query_start must start at 0, never decrease and end within the T rows
  if (blockIdx.x == 0 && warp == 0) {
    bool bad = lane == 0 && __ldg(p.query_start) != 0;
    for (int b = lane; b < p.B; b += 32) {
      const int s0 = __ldg(p.query_start + b), s1 = __ldg(p.query_start + b + 1);
      bad |= s1 < s0 || s1 > p.T;
    }
    if (__any_sync(kFull, bad) && lane == 0) record_error(p.err, kDevErrQuery);
  }

  // ---- the sequence and first query token of this tile (every warp finds the same)
  int b = -1, i0 = 0;
  {
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
        const int v = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += v;
      }
      const int total = __shfl_sync(kFull, incl, 31);
      if (tile_id < base + total) {
        const int first = __ffs(__ballot_sync(kFull, tile_id < base + incl)) - 1;
        const int before = __shfl_sync(kFull, incl - nt, first);
        b = b0 + first;
        i0 = (tile_id - base - before) * QT;
        break;
      }
      base += total;
    }
  }
  if (b < 0) return;  // past the last tile

  const int q0 = __ldg(p.query_start + b);
  const int n = __ldg(p.query_start + b + 1) - q0;
  const int L = __ldg(p.context_lens + b);
  if (L < 0 || L > p.MB * kBlockSize || n > L || q0 < 0 || q0 + n > p.T) {
    if (threadIdx.x == 0) record_error(p.err, (L < 0 || L > p.MB * kBlockSize) ? kDevErrLength : kDevErrQuery);
    return;
  }
  const int pos0 = L - n + i0;                         // position of the tile's first query token
  const int p_max = pos0 + min(QT, n - i0) - 1;        // of its last (<= L - 1)
  const int nkv = p_max / kKvTokens + 1;               // stages up to and including p_max

  extern __shared__ unsigned char smem_raw[];
  unsigned char* ring = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  const uint32_t ring_s = smem_addr(ring);
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + kPfStages * STAGE);
  uint64_t* empty = full + kPfStages;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kPfStages; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, kPfWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kPfWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const int32_t* row = p.block_tables + static_cast<int64_t>(b) * p.bt_sb;
      int slot = 0;
      uint32_t phase = 0;
      for (int j = 0; j < nkv; ++j) {
        if (j >= kPfStages) mbar_wait(empty + slot, phase ^ 1u, p.err);  // stage released
        int pb[2];
        uint32_t bytes = 0;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int jb = 2 * j + u;
          pb[u] = -1;
          if (jb * kBlockSize <= p_max) {
            const int e = __ldg(row + jb);
            if (static_cast<unsigned>(e) < static_cast<unsigned>(p.NB)) {
              pb[u] = e;
              bytes += 2 * TILE;
            } else {
              record_error(p.err, kDevErrBlockId);
            }
          }
        }
        if (bytes) {
          mbar_arrive_expect_tx(full + slot, bytes);
          unsigned char* st = ring + slot * STAGE;
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            if (pb[u] < 0) continue;
#pragma unroll
            for (int c = 0; c < BOXES; ++c) {
              tma_load_4d(st + u * TILE + c * kBoxBytes, &tmk, c * kBoxDims, 0, g, pb[u], full + slot);
              tma_load_4d(st + (2 + u) * TILE + c * kBoxBytes, &tmv, c * kBoxDims, 0, g, pb[u], full + slot);
            }
          }
        } else {
          mbar_arrive(full + slot);  // nothing to copy (a bad id is recorded above)
        }
        if (++slot == kPfStages) {
          slot = 0;
          phase ^= 1u;
        }
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int tq = lane >> 2, tr = lane & 3;
  const int r0 = warp * 16 + tq, r1 = r0 + 8;           // this thread's two rows of the tile
  const int tok0 = r0 / G, tok1 = r1 / G;               // their query tokens, from i0
  const int h0 = g * G + r0 % G, h1 = g * G + r1 % G;   // and heads
  const bool ok0 = i0 + tok0 < n, ok1 = i0 + tok1 < n;
  const int lim0 = ok0 ? pos0 + tok0 : p_max;           // causal limit of each row
  const int lim1 = ok1 ? pos0 + tok1 : p_max;

  // A operand Q (rows x dims): {row r0, dims 16ks + 2tr, +1}, {r1, same},
  // {r0, 16ks + 8 + 2tr, +1}, {r1, same}; rows past the run are 0.
  uint32_t qa[KSTEPS][4];
  {
    const __nv_bfloat16* qp0 = p.q + static_cast<int64_t>(q0 + i0 + tok0) * p.q_st + static_cast<int64_t>(h0) * p.q_sh;
    const __nv_bfloat16* qp1 = p.q + static_cast<int64_t>(q0 + i0 + tok1) * p.q_st + static_cast<int64_t>(h1) * p.q_sh;
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
      qa[ks][0] = ok0 ? ldg_u32(qp0 + 16 * ks + 2 * tr) : 0u;
      qa[ks][1] = ok1 ? ldg_u32(qp1 + 16 * ks + 2 * tr) : 0u;
      qa[ks][2] = ok0 ? ldg_u32(qp0 + 16 * ks + 8 + 2 * tr) : 0u;
      qa[ks][3] = ok1 ? ldg_u32(qp1 + 16 * ks + 8 + 2 * tr) : 0u;
    }
  }

  float o[D / 8][4];
#pragma unroll
  for (int dt = 0; dt < D / 8; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // running max (log2 units) and sum per row

  const int krow = (lane & 7) + ((lane >> 4) & 1) * 8;  // ldmatrix row addresses: K (B operand)
  const int kchunk = (lane >> 3) & 1;
  const int vrow = (lane & 7) + ((lane >> 3) & 1) * 8;  // V (B operand, transposed)
  const int vchunk = lane >> 4;

  int slot = 0;
  uint32_t phase = 0;
  for (int j = 0; j < nkv; ++j) {
    mbar_wait(full + slot, phase, p.err);
    unsigned char* st = ring + slot * STAGE;
    const uint32_t st_s = ring_s + slot * STAGE;
    const int t0 = j * kKvTokens;

    if (j == nkv - 1) {
      // V rows from z0 on may hold anything: past the sequence, or a block not loaded
      const int loaded_end = t0 + ((2 * j + 1) * kBlockSize <= p_max ? kKvTokens : kBlockSize);
      const int z0 = min(L, loaded_end) - t0;
      if (z0 < kKvTokens) {  // the same for every consumer warp
        for (int idx = threadIdx.x; idx < (kKvTokens - z0) * BOXES * 8; idx += kPfConsumers) {
          const int r = z0 + idx / (BOXES * 8), rest = idx % (BOXES * 8);
          *reinterpret_cast<uint4*>(st + (2 + (r >> 4)) * TILE + (rest >> 3) * kBoxBytes + (r & 15) * 128 +
                                    (rest & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        named_barrier(1, kPfConsumers);
      }
    }

    // ---- S = Q K^T: 16 rows x 32 tokens (n-tiles of 8 tokens)
    float s[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        uint32_t r[4];
        ldsm_x4(swz(st_s + u * TILE, krow, 2 * ks + kchunk), r);
        mma_16816_bf16(s[2 * u], qa[ks], r[0], r[1]);
        mma_16816_bf16(s[2 * u + 1], qa[ks], r[2], r[3]);
      }
    }

    // ---- causal mask, log2 units, running max and rescale
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int t = t0 + nt * 8 + 2 * tr + e;
        s[nt][e] = t <= lim0 ? s[nt][e] * p.qk_scale_log2 : -INFINITY;
        s[nt][2 + e] = t <= lim1 ? s[nt][2 + e] * p.qk_scale_log2 : -INFINITY;
        mx0 = fmaxf(mx0, s[nt][e]);
        mx1 = fmaxf(mx1, s[nt][2 + e]);
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 2));
    // every row sees token 0 in the first stage, so the running max is finite from then on
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float a0 = fast_exp2(m0 - mn0), a1 = fast_exp2(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    l0 *= a0;
    l1 *= a1;
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt) {
      o[dt][0] *= a0;
      o[dt][1] *= a0;
      o[dt][2] *= a1;
      o[dt][3] *= a1;
    }
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      s[nt][0] = fast_exp2(s[nt][0] - mn0);
      s[nt][1] = fast_exp2(s[nt][1] - mn0);
      s[nt][2] = fast_exp2(s[nt][2] - mn1);
      s[nt][3] = fast_exp2(s[nt][3] - mn1);
      l0 += s[nt][0] + s[nt][1];
      l1 += s[nt][2] + s[nt][3];
    }

    // ---- O += P V: k = 16 tokens per step (one block), P as bf16 hi + lo
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      uint32_t ah[4], al[4];
      split_bf16x2(s[2 * kk][0], s[2 * kk][1], ah[0], al[0]);
      split_bf16x2(s[2 * kk][2], s[2 * kk][3], ah[1], al[1]);
      split_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1], ah[2], al[2]);
      split_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3], ah[3], al[3]);
      const uint32_t vt = st_s + (2 + kk) * TILE;
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        uint32_t r[4];
        ldsm_x4_trans(swz(vt, vrow, 2 * dp + vchunk), r);
        mma_16816_bf16(o[2 * dp], ah, r[0], r[1]);
        mma_16816_bf16(o[2 * dp], al, r[0], r[1]);
        mma_16816_bf16(o[2 * dp + 1], ah, r[2], r[3]);
        mma_16816_bf16(o[2 * dp + 1], al, r[2], r[3]);
      }
    }

    __syncwarp();
    if (lane == 0) mbar_arrive(empty + slot);
    if (++slot == kPfStages) {
      slot = 0;
      phase ^= 1u;
    }
  }

  // ---- normalise and write this thread's two rows
  l0 += __shfl_xor_sync(kFull, l0, 1);
  l0 += __shfl_xor_sync(kFull, l0, 2);
  l1 += __shfl_xor_sync(kFull, l1, 1);
  l1 += __shfl_xor_sync(kFull, l1, 2);
  const float inv0 = 1.f / l0, inv1 = 1.f / l1;
  OutT* out0 = reinterpret_cast<OutT*>(p.out) + static_cast<int64_t>(q0 + i0 + tok0) * p.o_st +
               static_cast<int64_t>(h0) * p.o_sh;
  OutT* out1 = reinterpret_cast<OutT*>(p.out) + static_cast<int64_t>(q0 + i0 + tok1) * p.o_st +
               static_cast<int64_t>(h1) * p.o_sh;
#pragma unroll
  for (int dt = 0; dt < D / 8; ++dt) {
    const int d = 8 * dt + 2 * tr;
    if (ok0) store2(out0 + d, o[dt][0] * inv0, o[dt][1] * inv0);
    if (ok1) store2(out1 + d, o[dt][2] * inv1, o[dt][3] * inv1);
  }
}

// Raise the kernel's dynamic shared-memory limit once per device.
template <typename K>
cudaError_t ensure_prefill_smem(K kernel, size_t bytes, std::atomic<int> (&done)[64]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) dev = 63;
  if (done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess) done[dev].store(1);
  return e;
}

template <int D, int G, typename OutT>
cudaError_t launch_prefill_typed(const PrefillParams& p, const CUtensorMap& tmk, const CUtensorMap& tmv,
                                 cudaStream_t stream) {
  constexpr int QT = kPfRows / G;
  auto kernel = paged_prefill_kernel<D, G, OutT>;
  static std::atomic<int> smem_set[64];  // one record per instantiation
  const size_t smem = prefill_smem_bytes(D);
  cudaError_t e = ensure_prefill_smem(kernel, smem, smem_set);
  if (e != cudaSuccess) return e;
  // sum over sequences of ceil(n_b / QT) <= T / QT + B tiles
  const int64_t tiles = (static_cast<int64_t>(p.T) + QT - 1) / QT + p.B;
  if (tiles * p.Hkv > 0x7fffffff) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(tiles * p.Hkv));
  kernel<<<grid, kPfThreads, smem, stream>>>(tmk, tmv, p);
  return cudaGetLastError();
}

template <int D, typename OutT>
cudaError_t launch_prefill_g(const PrefillParams& p, const CUtensorMap& tmk, const CUtensorMap& tmv, int G,
                             cudaStream_t stream) {
  switch (G) {
    case 1: return launch_prefill_typed<D, 1, OutT>(p, tmk, tmv, stream);
    case 2: return launch_prefill_typed<D, 2, OutT>(p, tmk, tmv, stream);
    case 4: return launch_prefill_typed<D, 4, OutT>(p, tmk, tmv, stream);
    case 8: return launch_prefill_typed<D, 8, OutT>(p, tmk, tmv, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tmk, const CUtensorMap& tmv, int D, int G,
                           bool out_bf16, cudaStream_t stream) {
  if (p.B == 0 || p.T == 0) return cudaSuccess;
  if (D == 128) {
    return out_bf16 ? launch_prefill_g<128, __nv_bfloat16>(p, tmk, tmv, G, stream)
                    : launch_prefill_g<128, float>(p, tmk, tmv, G, stream);
  }
  if (D == 64) {
    return out_bf16 ? launch_prefill_g<64, __nv_bfloat16>(p, tmk, tmv, G, stream)
                    : launch_prefill_g<64, float>(p, tmk, tmv, G, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace forge
