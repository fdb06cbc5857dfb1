// Paged grouped-query-attention decode: one query token per sequence.
//
// forge-engine README, "What it implements", row "Kernels": decode attention
// over the paged KV cache is a CUDA paged GQA kernel.  "Make the Engine
// Talk", 1.2-1.3: decode runs one new token per sequence against everything
// cached so far, with grouped-query attention.  For query head h of sequence
// b, with G = Hq / Hkv and L = context_lens[b]:
//   out[b,h,:] = sum_{t<L} softmax_t(scale * q[b,h,:] . K[t, h/G, :]) V[t, h/G, :]
// where token t lives in physical block block_tables[b][t/16], slot t%16.
//
// Work decomposition (HBM-bound: ~2 fp32 FMA per byte of K/V at G = 4):
//   * one CTA per (split, KV head g, sequence b).  A split is a run of up to
//     `bps` consecutive KV blocks of one sequence; every K/V byte is read once
//     and used for all G query heads of its group;
//   * warp 4 is the producer: it translates logical blocks through the block
//     table and streams the split's K tiles, then its V tiles, into a ring of
//     shared-memory stages.  A stage holds two (block, head) tiles (16 x D
//     bf16 each, one contiguous run apiece), moved by single bulk copies on
//     the TMA engine and tracked by one mbarrier;
//   * warps 0-3 consume: 8 lanes per token, D/8 dims per lane, two tokens
//     per thread per stage.  Pass 1 forms the G logits of every token of the
//     split (packed fp32x2 FMA on bf16 widened exactly) and sums each 8-lane
//     group with a transposing shuffle reduction that ends with one (token,
//     head) logit per lane; the split's max and sum are then taken over all
//     logits at once (no running rescale); pass 2 accumulates p * V in
//     registers;
//   * a split that is the whole sequence writes `out` directly; otherwise it
//     writes unnormalised (acc, max, sum) and the reduce kernel merges the
//     splits of each (b, h).
// Logits are kept in log2 units (q is prescaled by scale*log2 e) so that the
// exponentials are single ex2 instructions.  Slots at t >= L are never
// multiplied in: their logits are -inf and their V rows are skipped, so NaN
// in unused slots cannot leak into the output.
#include <algorithm>
#include <atomic>
#include <cmath>

#include "common.cuh"

namespace forge {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kStageBlocks = 2;            // KV blocks per pipeline stage
constexpr int kGroups = kConsumers / 8;    // token groups (8 lanes each)

struct SmemLayout {
  size_t ring, logits, red_ml, bars, total;
};

// ring: nstage stages of kStageBlocks tiles; reused at the end for the
// cross-group sum, [kGroups][G][D] fp32.  logits: [bps*16][G] fp32 (rounded
// up to whole stages).
__host__ __device__ inline SmemLayout decode_layout(int D, int G, int bps, int nstage) {
  SmemLayout l;
  size_t off = 0;
  l.ring = off;
  const size_t ring = static_cast<size_t>(nstage) * kStageBlocks * kBlockSize * D * 2;
  const size_t red = static_cast<size_t>(kGroups) * G * D * 4;
  off += ring > red ? ring : red;
  l.logits = off;
  const int bps_up = (bps + kStageBlocks - 1) / kStageBlocks * kStageBlocks;
  off += static_cast<size_t>(bps_up) * kBlockSize * G * 4;
  l.red_ml = off;
  off += static_cast<size_t>(2) * kConsumerWarps * G * 4;
  off = (off + 15) & ~static_cast<size_t>(15);
  l.bars = off;
  off += static_cast<size_t>(2) * nstage * 8;
  l.total = off;
  return l;
}

template <int G>
__device__ __forceinline__ void load_row(const float* src, float (&v)[G]) {
  if constexpr (G % 4 == 0) {
#pragma unroll
    for (int k = 0; k < G / 4; ++k) {
      const float4 t = reinterpret_cast<const float4*>(src)[k];
      v[4 * k] = t.x;
      v[4 * k + 1] = t.y;
      v[4 * k + 2] = t.z;
      v[4 * k + 3] = t.w;
    }
  } else if constexpr (G == 2) {
    const float2 t = *reinterpret_cast<const float2*>(src);
    v[0] = t.x;
    v[1] = t.y;
  } else {
    v[0] = *src;
  }
}

template <int G>
__device__ __forceinline__ void store_row(float* dst, const float (&v)[G]) {
  if constexpr (G % 4 == 0) {
#pragma unroll
    for (int k = 0; k < G / 4; ++k)
      reinterpret_cast<float4*>(dst)[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
  } else if constexpr (G == 2) {
    *reinterpret_cast<float2*>(dst) = make_float2(v[0], v[1]);
  } else {
    *dst = v[0];
  }
}

__device__ __forceinline__ void store_out(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// Clamp a sequence length to what its block-table row can address; record a
// device error when the caller broke that precondition.
__device__ __forceinline__ int checked_length(const DecodeParams& p, int b, bool report) {
  int L = __ldg(p.context_lens + b);
  const int Lmax = p.MB * kBlockSize;
  if (L < 0 || L > Lmax) {
    if (report) record_error(p.err, kDevErrLength);
    L = L < 0 ? 0 : Lmax;
  }
  return L;
}

// Sum each of a lane's CNT values over the 8 lanes of its token group (lanes
// that differ in bits 0..2).  At each exchange step a lane keeps one half of
// the values it still holds and hands the other half to its partner, so the
// shuffle count halves per step.  Afterwards lane `sub` holds the group sums
// of values [first, first + max(N/8, 1)), returned in v[0..].
template <int CNT, int M>
struct Group8Sum {
  template <int N>
  static __device__ __forceinline__ void run(float (&v)[N], int sub, int& first) {
    const bool hi = (sub & M) != 0;
    if constexpr (CNT > 1) {
      constexpr int H = CNT / 2;
#pragma unroll
      for (int k = 0; k < H; ++k) {
        const float keep = hi ? v[H + k] : v[k];
        const float send = hi ? v[k] : v[H + k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, M);
      }
      if (hi) first += H;
      if constexpr (M > 1) Group8Sum<H, M / 2>::run(v, sub, first);
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], M);
      if constexpr (M > 1) Group8Sum<1, M / 2>::run(v, sub, first);
    }
  }
};

// Load one token row slice: chunk c (16 bytes) of this lane sits at element
// c * 64 + sub * 8, so the 8 lanes of a token read 128 contiguous bytes per
// chunk (no shared-memory bank conflicts).
template <int D>
__device__ __forceinline__ void load_row_slice(const __nv_bfloat16* row, int sub, uint32_t (&w)[D / 16]) {
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    const uint4 x = *reinterpret_cast<const uint4*>(row + c * 64 + sub * 8);
    w[4 * c] = x.x;
    w[4 * c + 1] = x.y;
    w[4 * c + 2] = x.z;
    w[4 * c + 3] = x.w;
  }
}

template <int D, int G, typename OutT>
__global__ void __launch_bounds__(kThreads, (G >= 8 ? 1 : 4)) paged_gqa_decode_split_kernel(const DecodeParams p) {
  constexpr int WPL = D / 16;  // bf16 pairs per lane per token row
  constexpr int TILE = kBlockSize * D;
  constexpr uint32_t kTileBytes = TILE * sizeof(__nv_bfloat16);
  constexpr int NV = kStageBlocks * G;  // logits a thread forms per stage
  static_assert(D % 64 == 0, "8 lanes x whole 16-byte chunks per token row");

  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int L = checked_length(p, b, s == 0 && g == 0 && threadIdx.x == 0);
  const int nblk = (L + kBlockSize - 1) / kBlockSize;
  const int nsplit = (nblk + p.bps - 1) / p.bps;

  if (L == 0) {  // empty context: the output is defined as zero
    if (s == 0) {
      for (int o = threadIdx.x; o < G * D; o += kThreads) {
        const int i = o / D, d = o % D;
        store_out(reinterpret_cast<OutT*>(p.out) + b * p.o_sb + (g * G + i) * p.o_sh + d, 0.f);
      }
    }
    return;
  }
  if (s >= nsplit) return;

  const int blk0 = s * p.bps;
  const int n = min(p.bps, nblk - blk0);                    // KV blocks in this split (>= 1)
  const int nks = (n + kStageBlocks - 1) / kStageBlocks;    // stages per pass
  const int nstage = p.nstage;

  extern __shared__ __align__(128) unsigned char smem[];
  const SmemLayout lay = decode_layout(D, G, p.bps, nstage);
  __nv_bfloat16* ring = reinterpret_cast<__nv_bfloat16*>(smem + lay.ring);
  float* red = reinterpret_cast<float*>(smem + lay.ring);  // reuses the ring at the end
  float* logits = reinterpret_cast<float*>(smem + lay.logits);
  float* red_m = reinterpret_cast<float*>(smem + lay.red_ml);
  float* red_l = red_m + kConsumerWarps * G;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.bars);
  uint64_t* empty = full + nstage;

  if (threadIdx.x == 0) {
    for (int i = 0; i < nstage; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, kConsumerWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    const int32_t* row = p.block_tables + static_cast<int64_t>(b) * p.bt_sb + blk0;
    const int e0 = lane < n ? __ldg(row + lane) : 0;
    const int e1 = lane + 32 < n ? __ldg(row + 32 + lane) : 0;
    const bool bad = (lane < n && static_cast<unsigned>(e0) >= static_cast<unsigned>(p.NB)) ||
                     (lane + 32 < n && static_cast<unsigned>(e1) >= static_cast<unsigned>(p.NB));
    if (__any_sync(0xffffffffu, bad) && lane == 0) record_error(p.err, kDevErrBlockId);
    const __nv_bfloat16* kbase = p.k_cache + g * p.kc_sh;
    const __nv_bfloat16* vbase = p.v_cache + g * p.vc_sh;
    int slot = 0;
    uint32_t phase = 0;
    for (int i = 0; i < 2 * nks; ++i) {
      const bool is_v = i >= nks;
      const int j0 = (is_v ? i - nks : i) * kStageBlocks;
      int pb[kStageBlocks];
#pragma unroll
      for (int u = 0; u < kStageBlocks; ++u) {
        const int j = j0 + u;  // <= 63 < 2 * 32
        pb[u] = __shfl_sync(0xffffffffu, j < 32 ? e0 : e1, j & 31);
        if (j >= n) pb[u] = -1;  // past the split: no tile
      }
      if (lane == 0) {
        if (i >= nstage) mbar_wait(empty + slot, phase ^ 1u, p.err);  // stage released
        uint32_t bytes = 0;
#pragma unroll
        for (int u = 0; u < kStageBlocks; ++u)
          if (static_cast<unsigned>(pb[u]) < static_cast<unsigned>(p.NB)) bytes += kTileBytes;
        if (bytes) {
          mbar_arrive_expect_tx(full + slot, bytes);
          const __nv_bfloat16* base = is_v ? vbase : kbase;
          const int64_t sblk = is_v ? p.vc_sblk : p.kc_sblk;
#pragma unroll
          for (int u = 0; u < kStageBlocks; ++u)
            if (static_cast<unsigned>(pb[u]) < static_cast<unsigned>(p.NB))
              bulk_copy_g2s(ring + (slot * kStageBlocks + u) * TILE, base + static_cast<int64_t>(pb[u]) * sblk,
                            kTileBytes, full + slot);
        } else {
          mbar_arrive(full + slot);  // nothing to copy (bad ids are recorded above)
        }
      }
      if (++slot == nstage) {
        slot = 0;
        phase ^= 1u;
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int tid = threadIdx.x;  // 0 .. kConsumers-1
  const int tok = tid >> 3;     // token row within each tile of a stage
  const int sub = tid & 7;
  const int t_base = blk0 * kBlockSize;

  // q of the G heads of this group, prescaled into log2 units, as float pairs
  // in this lane's dims {c*64 + sub*8 + e}.
  float2 q2[G][WPL];
#pragma unroll
  for (int i = 0; i < G; ++i) {
    uint32_t w[WPL];
    load_row_slice<D>(p.q + static_cast<int64_t>(b) * p.q_sb + static_cast<int64_t>(g * G + i) * p.q_sh, sub, w);
#pragma unroll
    for (int k = 0; k < WPL; ++k) {
      const float2 f = bf16x2_to_float2(w[k]);
      q2[i][k] = make_float2(f.x * p.qk_scale_log2, f.y * p.qk_scale_log2);
    }
  }

  int slot = 0;
  uint32_t phase = 0;

  // ---- pass 1: logits of every token of the split (log2 units)
  for (int st = 0; st < nks; ++st) {
    mbar_wait(full + slot, phase, p.err);
    float v[NV];
#pragma unroll
    for (int u = 0; u < kStageBlocks; ++u) {
      uint32_t kw[WPL];
      load_row_slice<D>(ring + (slot * kStageBlocks + u) * TILE + tok * D, sub, kw);
      if (u == kStageBlocks - 1) {
        __syncwarp();
        if (lane == 0) mbar_arrive(empty + slot);
      }
      float2 acc[G];
#pragma unroll
      for (int i = 0; i < G; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < WPL; ++k) {
        const float2 kf = bf16x2_to_float2(kw[k]);
#pragma unroll
        for (int i = 0; i < G; ++i) acc[i] = ffma2(q2[i][k], kf, acc[i]);
      }
#pragma unroll
      for (int i = 0; i < G; ++i) v[u * G + i] = acc[i].x + acc[i].y;
    }
    int first = 0;
    Group8Sum<NV, 4>::run(v, sub, first);
    constexpr int kOut = NV >= 8 ? NV / 8 : 1;
    constexpr int kDup = NV >= 8 ? 1 : 8 / NV;  // lanes holding the same sum
    if ((sub & (kDup - 1)) == 0) {
#pragma unroll
      for (int k = 0; k < kOut; ++k) {
        const int idx = first + k;
        const int u = idx / G, i = idx % G;
        const int j = st * kStageBlocks + u;  // block within the split
        if (j < n) {
          const bool valid = t_base + j * kBlockSize + tok < L;
          logits[(j * kBlockSize + tok) * G + i] = valid ? v[k] : -INFINITY;
        }
      }
    }
    if (++slot == nstage) {
      slot = 0;
      phase ^= 1u;
    }
  }
  named_barrier(1, kConsumers);

  // ---- softmax over the split: max, then p = 2^(s - max) in place, and sum
  const int ntok = n * kBlockSize;
  {
    float mx[G];
#pragma unroll
    for (int i = 0; i < G; ++i) mx[i] = -INFINITY;
    for (int t = tid; t < ntok; t += kConsumers) {
      float x[G];
      load_row<G>(logits + t * G, x);
#pragma unroll
      for (int i = 0; i < G; ++i) mx[i] = fmaxf(mx[i], x[i]);
    }
#pragma unroll
    for (int i = 0; i < G; ++i) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], off));
    }
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < G; ++i) red_m[warp * G + i] = mx[i];
    }
    named_barrier(1, kConsumers);
    float m[G];
#pragma unroll
    for (int i = 0; i < G; ++i) {
      m[i] = red_m[i];
#pragma unroll
      for (int w = 1; w < kConsumerWarps; ++w) m[i] = fmaxf(m[i], red_m[w * G + i]);
    }
    float sum[G];
#pragma unroll
    for (int i = 0; i < G; ++i) sum[i] = 0.f;
    for (int t = tid; t < ntok; t += kConsumers) {
      float x[G];
      load_row<G>(logits + t * G, x);
#pragma unroll
      for (int i = 0; i < G; ++i) {
        x[i] = fast_exp2(x[i] - m[i]);
        sum[i] += x[i];
      }
      store_row<G>(logits + t * G, x);
    }
#pragma unroll
    for (int i = 0; i < G; ++i) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum[i] += __shfl_xor_sync(0xffffffffu, sum[i], off);
    }
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < G; ++i) red_l[warp * G + i] = sum[i];
    }
    named_barrier(1, kConsumers);
  }

  // ---- pass 2: acc += p * V over this thread's tokens
  float2 acc[G][WPL];
#pragma unroll
  for (int i = 0; i < G; ++i)
#pragma unroll
    for (int k = 0; k < WPL; ++k) acc[i][k] = make_float2(0.f, 0.f);

  for (int st = 0; st < nks; ++st) {
    mbar_wait(full + slot, phase, p.err);
    uint32_t vw[kStageBlocks][WPL];
#pragma unroll
    for (int u = 0; u < kStageBlocks; ++u)
      load_row_slice<D>(ring + (slot * kStageBlocks + u) * TILE + tok * D, sub, vw[u]);
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + slot);
#pragma unroll
    for (int u = 0; u < kStageBlocks; ++u) {
      const int j = st * kStageBlocks + u;
      if (j < n && t_base + j * kBlockSize + tok < L) {
        float w[G];
        load_row<G>(logits + (j * kBlockSize + tok) * G, w);
#pragma unroll
        for (int k = 0; k < WPL; ++k) {
          const float2 vf = bf16x2_to_float2(vw[u][k]);
#pragma unroll
          for (int i = 0; i < G; ++i) acc[i][k] = ffma2(make_float2(w[i], w[i]), vf, acc[i][k]);
        }
      }
    }
    if (++slot == nstage) {
      slot = 0;
      phase ^= 1u;
    }
  }

  // ---- combine the kGroups token groups through shared memory (the ring is
  // free: every stage has been consumed by all consumer warps)
  named_barrier(1, kConsumers);
#pragma unroll
  for (int i = 0; i < G; ++i)
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      float4* dst = reinterpret_cast<float4*>(red + (tok * G + i) * D + c * 64 + sub * 8);
      dst[0] = make_float4(acc[i][4 * c].x, acc[i][4 * c].y, acc[i][4 * c + 1].x, acc[i][4 * c + 1].y);
      dst[1] = make_float4(acc[i][4 * c + 2].x, acc[i][4 * c + 2].y, acc[i][4 * c + 3].x, acc[i][4 * c + 3].y);
    }
  named_barrier(1, kConsumers);

  for (int o = tid * 4; o < G * D; o += kConsumers * 4) {
    const int i = o / D, d = o % D;
    float4 t = *reinterpret_cast<const float4*>(red + i * D + d);
#pragma unroll
    for (int grp = 1; grp < kGroups; ++grp) {
      const float4 x = *reinterpret_cast<const float4*>(red + (grp * G + i) * D + d);
      t.x += x.x;
      t.y += x.y;
      t.z += x.z;
      t.w += x.w;
    }
    // the split's sum for head i: total of the per-warp sums
    float li = red_l[i];
#pragma unroll
    for (int w = 1; w < kConsumerWarps; ++w) li += red_l[w * G + i];
    const int h = g * G + i;
    if (nsplit == 1) {
      OutT* dst = reinterpret_cast<OutT*>(p.out) + b * p.o_sb + h * p.o_sh + d;
      store_out(dst + 0, t.x / li);
      store_out(dst + 1, t.y / li);
      store_out(dst + 2, t.z / li);
      store_out(dst + 3, t.w / li);
    } else {
      *reinterpret_cast<float4*>(p.ws_acc + ((static_cast<int64_t>(b) * p.Hq + h) * p.s_max + s) * D + d) = t;
    }
  }
  if (nsplit > 1 && tid < G) {
    float mi = red_m[tid], li = red_l[tid];
#pragma unroll
    for (int w = 1; w < kConsumerWarps; ++w) {
      mi = fmaxf(mi, red_m[w * G + tid]);
      li += red_l[w * G + tid];
    }
    const int64_t r = (static_cast<int64_t>(b) * p.Hq + g * G + tid) * p.s_max + s;
    p.ws_ml[2 * r] = mi;
    p.ws_ml[2 * r + 1] = li;
  }
}

// Merge the split partials of every (b, h) whose sequence has more than one
// split: with M = max_s m_s and w_s = 2^(m_s - M),
//   out = sum_s w_s acc_s / sum_s w_s l_s.
// One warp per (b, h); each lane owns D/32 consecutive dims.  The split loop
// is unrolled by 8 so that eight partial rows are in flight at once.
template <int D, typename OutT>
__global__ void __launch_bounds__(128) paged_gqa_decode_reduce_kernel(const DecodeParams p) {
  constexpr int DPT = D / 32;
  constexpr int U = 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rowid = static_cast<int64_t>(blockIdx.x) * 4 + warp;
  if (rowid >= static_cast<int64_t>(p.B) * p.Hq) return;
  const int b = static_cast<int>(rowid / p.Hq), h = static_cast<int>(rowid % p.Hq);
  const int L = checked_length(p, b, false);
  const int nblk = (L + kBlockSize - 1) / kBlockSize;
  const int nsplit = (nblk + p.bps - 1) / p.bps;
  if (nsplit <= 1) return;

  const float* ml = p.ws_ml + rowid * p.s_max * 2;
  float M = -INFINITY;
  for (int s = lane; s < nsplit; s += 32) M = fmaxf(M, ml[2 * s]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float lsum = 0.f;
  for (int s = lane; s < nsplit; s += 32) lsum += fast_exp2(ml[2 * s] - M) * ml[2 * s + 1];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);

  float acc[DPT];
#pragma unroll
  for (int k = 0; k < DPT; ++k) acc[k] = 0.f;
  const float* a = p.ws_acc + rowid * p.s_max * D + lane * DPT;
  int s = 0;
  for (; s + U <= nsplit; s += U) {
    float x[U][DPT], w[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      w[u] = ml[2 * (s + u)];
      const float* src = a + static_cast<int64_t>(s + u) * D;
      if constexpr (DPT == 4) {
        const float4 t = *reinterpret_cast<const float4*>(src);
        x[u][0] = t.x;
        x[u][1] = t.y;
        x[u][2] = t.z;
        x[u][3] = t.w;
      } else {
        const float2 t = *reinterpret_cast<const float2*>(src);
        x[u][0] = t.x;
        x[u][1] = t.y;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float wu = fast_exp2(w[u] - M);
#pragma unroll
      for (int k = 0; k < DPT; ++k) acc[k] = fmaf(wu, x[u][k], acc[k]);
    }
  }
  for (; s < nsplit; ++s) {
    const float wu = fast_exp2(ml[2 * s] - M);
#pragma unroll
    for (int k = 0; k < DPT; ++k) acc[k] = fmaf(wu, a[static_cast<int64_t>(s) * D + k], acc[k]);
  }
  OutT* o = reinterpret_cast<OutT*>(p.out) + b * p.o_sb + h * p.o_sh + lane * DPT;
#pragma unroll
  for (int k = 0; k < DPT; ++k) store_out(o + k, acc[k] / lsum);
}

// Raise a kernel's dynamic shared-memory limit once per device and size.
// `set_for` is the caller's own per-kernel record of what it already set.
template <typename K>
cudaError_t ensure_smem(K kernel, size_t bytes, std::atomic<size_t> (&set_for)[64]) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) dev = 63;
  if (set_for[dev].load(std::memory_order_relaxed) >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess) {
    size_t cur = set_for[dev].load();
    while (cur < bytes && !set_for[dev].compare_exchange_weak(cur, bytes)) {
    }
  }
  return e;
}

template <int D, int G, typename OutT>
cudaError_t launch_typed(const DecodeParams& p, cudaStream_t stream) {
  const size_t smem = decode_layout(D, G, p.bps, p.nstage).total;
  auto split_kernel = paged_gqa_decode_split_kernel<D, G, OutT>;
  static std::atomic<size_t> smem_set[64];  // one record per instantiation
  cudaError_t e = ensure_smem(split_kernel, smem, smem_set);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(p.s_max), static_cast<unsigned>(p.Hkv), static_cast<unsigned>(p.B));
  split_kernel<<<grid, kThreads, smem, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess || p.s_max <= 1) return e;
  const int64_t rows = static_cast<int64_t>(p.B) * p.Hq;
  paged_gqa_decode_reduce_kernel<D, OutT><<<static_cast<unsigned>((rows + 3) / 4), 128, 0, stream>>>(p);
  return cudaGetLastError();
}

template <int D, typename OutT>
cudaError_t launch_g(const DecodeParams& p, int G, cudaStream_t stream) {
  switch (G) {
    case 1: return launch_typed<D, 1, OutT>(p, stream);
    case 2: return launch_typed<D, 2, OutT>(p, stream);
    case 4: return launch_typed<D, 4, OutT>(p, stream);
    case 8: return launch_typed<D, 8, OutT>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

size_t decode_smem_bytes(int D, int G, int bps, int nstage) {
  return decode_layout(D, G, bps, nstage).total;
}

cudaError_t launch_decode(const DecodeParams& p, int D, int G, bool out_bf16, cudaStream_t stream) {
  if (p.B == 0) return cudaSuccess;
  if (D == 128) {
    return out_bf16 ? launch_g<128, __nv_bfloat16>(p, G, stream) : launch_g<128, float>(p, G, stream);
  }
  if (D == 64) {
    return out_bf16 ? launch_g<64, __nv_bfloat16>(p, G, stream) : launch_g<64, float>(p, G, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace forge
