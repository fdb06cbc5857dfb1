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
// Work decomposition.  The path is HBM-bound (each K/V byte is used for G
// query heads); the kernel's job is to stream every byte once with as few
// SM instructions per byte as possible:
//   * one CTA per (KV head g, sequence b, split).  A split is a run of up to
//     `bps` consecutive KV blocks of one sequence;
//   * warp 2 is the producer: it translates logical blocks through the block
//     table and streams the split's K tiles, then its V tiles, into a ring of
//     shared-memory stages with tiled TMA copies (5-D tensor maps over the
//     cache, 128-byte swizzle, one copy per (block, head) tile, issued by the
//     lane of that tile).  A stage holds two tiles of 16 x D bf16 and is
//     tracked by one mbarrier;
//   * warps 0 and 1 consume one tile each per stage on the tensor cores
//     (mma.sync m16n8k16, bf16 in, fp32 accumulate; the G <= 8 query heads
//     fill the n = 8 side).  Pass 1: logits S^T = K q^T, 16 tokens per tile,
//     into shared memory in log2 units.  The split's max and sum are taken
//     over all its logits at once (no running rescale).  Pass 2:
//     O^T += V^T P^T with P split into bf16 high and low parts, so the
//     weights keep ~16 bits of precision; for G <= 4 the low parts ride in
//     the n columns no head uses, so this takes one MMA per 16 dims;
//   * a split that is the whole sequence writes `out` directly.  Otherwise
//     it writes unnormalised (acc, max, sum) to the workspace and counts
//     itself in at a per-(b, g) arrival counter; the CTA that arrives last
//     merges the splits of the G heads (the split reduce) and returns the
//     counter to zero.  Merging in the last CTA, rather than in a second
//     kernel, keeps the merge off the launch critical path.
// That is the two-pass kernel.  A second, single-pass kernel on the same grid
// (further below) carries K and V of the same blocks in each stage and keeps
// a running maximum and sum instead of a logits buffer, so all of its shared
// memory is K/V ring.  The host plan (abi.cu) runs the single-pass kernel
// unless FORGE_DECODE_KERNEL selects the two-pass one.
// Both are launched with programmatic stream serialization.  Before
// griddepcontrol.wait a CTA only reads its sequence length and block-table
// entries through L2 to prefetch its first K/V tiles into L2 (the values may
// be stale and steer nothing else); everything it uses is read after the wait.
// Slots at t >= L never reach the output: their logits are -inf and their V
// rows are zeroed in shared memory before the PV product, so NaN in unused
// slots cannot leak in.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <type_traits>

#include "common.cuh"

namespace forge {
namespace {

constexpr int kStageBlocks = 2;              // KV blocks (tiles) per pipeline stage
constexpr int kConsumerWarps = kStageBlocks; // one tile per consumer warp per stage
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;    // + one producer warp

// The n = 8 columns of the MMAs' B operands and accumulators (QK^T: the query
// heads; P V: the softmax weights of those heads).  With G <= 4 heads per
// group only columns 0-3 would carry heads, so column c holds head c % 4
// (when that head exists): the same q in columns c and c + 4 gives the same
// logits and weights there, and in P V columns 0-3 carry the weights' bf16
// high part and columns 4-7 their low part.  One MMA per 16 dims then gives P
// about 16 significant bits; the two halves of O are added once at the end.
// At G = 8 every column is a head and P V takes two MMAs (high, then low).
template <int G>
struct PvCols {
  static constexpr bool kPacked = G <= 4;
  __device__ static __forceinline__ int head(int c) { return kPacked ? (c & 3) : c; }
  __device__ static __forceinline__ bool valid(int c) { return head(c) < G; }
  __device__ static __forceinline__ bool low(int c) { return kPacked && c >= 4; }
};

// B fragment of P^T for column `col` of a P V MMA from four weights: the
// bf16 high parts, or for a packed low column the low parts (x - bf16(x)
// rounded to bf16); `lo*` receive the low parts for the second MMA at G = 8.
template <int G>
__device__ __forceinline__ void p_fragment(int col, float2 pa, float2 pc, uint32_t& b0, uint32_t& b1, uint32_t& lo0,
                                           uint32_t& lo1) {
  split_bf16x2(pa.x, pa.y, b0, lo0);
  split_bf16x2(pc.x, pc.y, b1, lo1);
  if (PvCols<G>::low(col)) {
    b0 = lo0;
    b1 = lo1;
  }
}

// Add each packed low column of the O^T accumulators into its high column
// (lanes 4 apart in the accumulator layout: column 2 (lane % 4) + e).
template <int G, int MT>
__device__ __forceinline__ void fold_low_columns(float (&o)[MT][4]) {
  if constexpr (PvCols<G>::kPacked) {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[mt][e] += __shfl_xor_sync(0xffffffffu, o[mt][e], 2);
  }
}

struct SmemLayout {
  size_t ring, logits, red_ml, bars, total;
  int lrow;  // logits row length (tokens) per head
};

// ring (1024-byte aligned for the 128-byte swizzle; reused at the end for the
// consumer-warp merge [kConsumerWarps][G][D] fp32) | logits [G][lrow] fp32 |
// per-warp (max, sum) | mbarriers.
__host__ __device__ inline SmemLayout decode_layout(int D, int G, int bps, int nstage) {
  SmemLayout l;
  size_t off = 1024;  // room to round the ring up to a 1024-byte boundary
  l.ring = off;
  const size_t ring = static_cast<size_t>(nstage) * kStageBlocks * kBlockSize * D * 2;
  const size_t red = static_cast<size_t>(kConsumerWarps) * G * D * 4;
  off += ring > red ? ring : red;
  l.logits = off;
  l.lrow = (bps + kStageBlocks - 1) / kStageBlocks * kStageBlocks * kBlockSize;
  off += static_cast<size_t>(G) * l.lrow * 4;
  l.red_ml = off;
  off += static_cast<size_t>(2) * kConsumerWarps * G * 4;
  off = (off + 15) & ~static_cast<size_t>(15);
  l.bars = off;
  off += static_cast<size_t>(2) * nstage * 8;
  l.total = off;
  return l;
}

__device__ __forceinline__ void store_out(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_out(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// Clamp a sequence length to what its block-table row can address; record a
// device error when the caller broke that precondition.
// A read-only load the compiler keeps where it is written (it is not sunk
// below the early exits that follow it), so that it overlaps other loads.
__device__ __forceinline__ int ld_nc_keep(const int32_t* ptr) {
  int v;
  asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(ptr));
  return v;
}

__device__ __forceinline__ int checked_length(const DecodeParams& p, int b, bool report) {
  int L = __ldg(p.context_lens + b);
  const int Lmax = p.MB * kBlockSize;
  if (L < 0 || L > Lmax) {
    if (report) record_error(p.err, kDevErrLength);
    L = L < 0 ? 0 : Lmax;
  }
  return L;
}

// A load through L2 only (no L1 copy), for values read before the previous
// grid in the stream has completed: they may be stale, and a later load of
// the same address must not find them in L1.
__device__ __forceinline__ int ld_cg(const int32_t* ptr) {
  int v;
  asm volatile("ld.global.cg.b32 %0, [%1];" : "=r"(v) : "l"(ptr));
  return v;
}

// Split s of a sequence of L tokens.  Splits are aligned to the END of the
// sequence: split nsplit-1 ends at its last block, every split but split 0
// holds bps blocks and split 0 the remaining r = nblk - (nsplit-1) bps (1..bps).
// The grid runs the highest split index first, so full splits are dispatched
// before the partial ones and the tail of the last wave is made of short CTAs
// (the longest-first order that evens out ragged batches).
struct SplitWork {
  int nblk, nsplit, blk0, n;
};
__device__ __forceinline__ SplitWork split_work(int L, int bps, int s) {
  SplitWork w;
  w.nblk = (L + kBlockSize - 1) / kBlockSize;
  w.nsplit = (w.nblk + bps - 1) / bps;
  const int r = w.nblk - (w.nsplit - 1) * bps;
  w.blk0 = s == 0 ? 0 : r + (s - 1) * bps;
  w.n = s == 0 ? r : bps;
  return w;
}

// The block-table entries of split s, requested by the producer warp before
// the length is known: for s >= 1 the split starts in [(s-1) bps + 1, s bps],
// so the 2 bps - 1 entries from w0 = (s-1) bps + 1 (from 0 for s = 0) cover
// it.  Lane l holds entries w0 + l + 32 k, k < 4 (bps <= 64); entries past
// the row are 0 and never used.
struct TableWindow {
  int e0, e1, e2, e3, w0;
  __device__ __forceinline__ void load(const DecodeParams& p, int b, int s, int lane) {
    w0 = s == 0 ? 0 : (s - 1) * p.bps + 1;
    const int32_t* row = p.block_tables + static_cast<int64_t>(b) * p.bt_sb;
    const int end = min(p.MB, w0 + 2 * p.bps - 1);
    const int i = w0 + lane;
    e0 = i < end ? ld_nc_keep(row + i) : 0;
    e1 = i + 32 < end ? ld_nc_keep(row + i + 32) : 0;
    e2 = i + 64 < end ? ld_nc_keep(row + i + 64) : 0;
    e3 = i + 96 < end ? ld_nc_keep(row + i + 96) : 0;
  }
  // the entry of block `blk` (warp-uniform) of the window, from its lane
  __device__ __forceinline__ int entry(int blk) const {
    const int i = blk - w0;
    const int k = i >> 5;
    return __shfl_sync(0xffffffffu, k == 0 ? e0 : k == 1 ? e1 : k == 2 ? e2 : e3, i & 31);
  }
  // any of the split's entries [blk0, blk0 + n) outside [0, NB)
  __device__ __forceinline__ bool any_bad(int blk0, int n, int NB, int lane) const {
    const int a = blk0 - w0, z = a + n;
    const int i = lane;
    const bool bad = (i >= a && i < z && static_cast<unsigned>(e0) >= static_cast<unsigned>(NB)) ||
                     (i + 32 >= a && i + 32 < z && static_cast<unsigned>(e1) >= static_cast<unsigned>(NB)) ||
                     (i + 64 >= a && i + 64 < z && static_cast<unsigned>(e2) >= static_cast<unsigned>(NB)) ||
                     (i + 96 >= a && i + 96 < z && static_cast<unsigned>(e3) >= static_cast<unsigned>(NB));
    return __any_sync(0xffffffffu, bad);
  }
};

// Before griddepcontrol.wait: bring the K and V tiles of the first `stages`
// ring stages of this CTA into L2 while the previous grid in the stream
// finishes.  The length and table entries are read through L2 only and may
// be stale: they steer prefetches alone (block ids are checked against the
// pool, and the TMA engine bounds-checks tensor coordinates); every value
// the kernel uses is read again after the wait.  One lane per block.
template <int D>
__device__ __forceinline__ void prefetch_first_stages(const CUtensorMap* tmk, const CUtensorMap* tmv,
                                                      const DecodeParams& p, int b, int g, int s, int stages,
                                                      int lane) {
  int L = ld_cg(p.context_lens + b);
  L = L < 0 ? 0 : min(L, p.MB * kBlockSize);
  const SplitWork w = split_work(L, p.bps, s);
  if (s >= w.nsplit || lane >= min(w.n, stages * 2)) return;
  const int pb = ld_cg(p.block_tables + static_cast<int64_t>(b) * p.bt_sb + w.blk0 + lane);
  if (static_cast<unsigned>(pb) >= static_cast<unsigned>(p.NB)) return;
  tma_prefetch_5d(tmk, 0, 0, 0, g, pb);
  tma_prefetch_5d(tmv, 0, 0, 0, g, pb);
}

// Fused append: put this step's new row (`src`, D bf16) into row `r` of the
// staged swizzled tile at `tile`, and into the cache row `cache_row` (when
// not null), 16 bytes per lane.  Then order the shared-memory writes before
// the warp's ldmatrix reads and before the TMA engine reuses the stage.
template <int D>
__device__ __forceinline__ void patch_new_row(unsigned char* tile, const __nv_bfloat16* src,
                                              __nv_bfloat16* cache_row, int r, int lane) {
  for (int c = lane; c < D / 8; c += 32) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(src) + c);
    *reinterpret_cast<uint4*>(tile + (c >> 3) * kBoxBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = v;
    if (cache_row) reinterpret_cast<uint4*>(cache_row)[c] = v;
  }
  fence_proxy_async_smem();
  __syncwarp();
}

// The q/k path ("Make the Engine Talk", 1.3: RMSNorm and rotary position
// embeddings), for the q fragments of one head held by the 4 lanes of an MMA
// group: x[ks][e] is dim 16 ks + 2 tr + e (e < 2) or 16 ks + 8 + 2 tr + e - 2
// (e >= 2).  RMSNorm with weight w_q (sum of squares over the 4 lanes), then
// rotate-half RoPE at `pos`: dim d < D/2 pairs with d + D/2, which is slot
// ks + D/32 of the same lane.  fp32 throughout.
template <int D>
__device__ __forceinline__ void q_norm_rope(float (&x)[D / 16][4], int tr, const DecodeParams& p, int pos,
                                            bool rope) {
  constexpr int K = D / 16;
  auto dim = [&](int ks, int e) { return 16 * ks + (e < 2 ? 2 * tr + e : 8 + 2 * tr + e - 2); };
  if (p.q_norm_w) {
    float ss = 0.f;
#pragma unroll
    for (int ks = 0; ks < K; ++ks)
#pragma unroll
      for (int e = 0; e < 4; ++e) ss = fmaf(x[ks][e], x[ks][e], ss);
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
    const float inv = rsqrtf(ss / D + p.norm_eps);
#pragma unroll
    for (int ks = 0; ks < K; ++ks)
#pragma unroll
      for (int e = 0; e < 4; ++e) x[ks][e] *= inv * __bfloat162float(p.q_norm_w[dim(ks, e)]);
  }
  if (rope) {
    const float* cs = p.rope + static_cast<int64_t>(pos) * D;
#pragma unroll
    for (int ks = 0; ks < K / 2; ++ks)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int d = dim(ks, e);
        const float c = __ldg(cs + d), sn = __ldg(cs + D / 2 + d);
        const float x1 = x[ks][e], x2 = x[ks + K / 2][e];
        x[ks][e] = x1 * c - x2 * sn;
        x[ks + K / 2][e] = x2 * c + x1 * sn;
      }
  }
}

// Fused append with the q/k path: the new K row (`src`) through RMSNorm
// (weight w_k) and RoPE at `pos`, rounded once to bf16, into row `r` of the
// staged tile and into the cache row.  Lane c < D/8 holds dims 8c .. 8c+7;
// its rotation partner (dims D/2 away) is lane c ^ (D/16).
template <int D>
__device__ __forceinline__ void patch_new_k_row(unsigned char* tile, const __nv_bfloat16* src,
                                                __nv_bfloat16* cache_row, int r, int lane, const DecodeParams& p,
                                                int pos, bool rope) {
  constexpr int C = D / 8;
  const bool has = lane < C;
  float x[8];
  if (has) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(src) + lane);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[2 * k] = bf16lo(w[k]);
      x[2 * k + 1] = bf16hi(w[k]);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = 0.f;
  }
  if (p.k_norm_w) {
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float inv = rsqrtf(ss / D + p.norm_eps);
    if (has) {
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] *= inv * __bfloat162float(p.k_norm_w[8 * lane + e]);
    }
  }
  if (rope) {
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = __shfl_xor_sync(0xffffffffu, x[e], C / 2);
    if (has) {
      const bool first = lane < C / 2;
      const int d0 = 8 * (first ? lane : lane - C / 2);  // rotation index of this lane's dims
      const float* cs = p.rope + static_cast<int64_t>(pos) * D;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float c = __ldg(cs + d0 + e), sn = __ldg(cs + D / 2 + d0 + e);
        x[e] = first ? x[e] * c - y[e] * sn : x[e] * c + y[e] * sn;
      }
    }
  }
  if (has) {
    const uint4 v = make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                               pack_bf16x2(x[6], x[7]));
    *reinterpret_cast<uint4*>(tile + (lane >> 3) * kBoxBytes + r * 128 + (((lane & 7) ^ (r & 7)) << 4)) = v;
    if (cache_row) reinterpret_cast<uint4*>(cache_row)[lane] = v;
  }
  fence_proxy_async_smem();
  __syncwarp();
}

// Split reduce for the G heads of (b, g): with M = max_s m_s and
// w_s = 2^(m_s - M), out = sum_s w_s acc_s / sum_s w_s l_s over the nsplit
// partials in the workspace.  Run by the kConsumers threads of the last CTA,
// in shared memory the CTA no longer needs (`wbuf`, wcap floats, 16-byte
// aligned).  Each L2 round trip here sits on the kernel's tail, so a chunk of
// up to cap splits is fetched at once: every thread copies the partial rows
// of the outputs it owns (4 consecutive dims each) straight into shared
// memory with asynchronous copies, all in flight together, while the
// chunk's (m, l) pairs are read ([G][cap] float2).  Each thread then takes
// its heads' maximum over the chunk and accumulates its outputs from its own
// copies; a running maximum carries across chunks (the sums are rescaled
// when it grows).  Workspace reads bypass L1 (other SMs wrote them).
// The callers' buffers hold at least 3 splits per chunk: both pass a region
// that contains the K/V ring, at least 2 stages of 2 K tiles, 128 D bytes,
// and a split takes (G D + 2 G) * 4 <= 36 D bytes.
template <int D, int G, typename OutT>
__device__ __forceinline__ void merge_splits(const DecodeParams& p, int b, int g, int nsplit, int tid, float* wbuf,
                                             int wcap) {
  constexpr int kRow4 = G * D / 4;                               // float4 outputs of the group
  constexpr int kOut = (kRow4 + kConsumers - 1) / kConsumers;    // float4 outputs per thread
  constexpr bool kEven = kRow4 % kConsumers == 0;                // every thread owns kOut outputs
  const int64_t row0 = static_cast<int64_t>(b) * p.Hq + g * G;  // first head of the group
  const int cap = wcap / (G * D + 2 * G);                        // splits per chunk
  float4* rows = reinterpret_cast<float4*>(wbuf);                // [cap][kRow4]
  float2* mlb = reinterpret_cast<float2*>(wbuf + static_cast<size_t>(cap) * G * D);  // [G][cap]
  const float2* ws_ml = reinterpret_cast<const float2*>(p.ws_ml);

  // output k of this thread: float4 o = tid + k * kConsumers of the group,
  // head o / (D / 4), dims 4 * (o % (D / 4))
  auto valid = [&](int k) { return kEven || tid + k * kConsumers < kRow4; };
  auto head = [&](int k) { return (tid + k * kConsumers) / (D / 4); };
  auto acc = [&](int k, int sp) {
    const int o4 = (tid + k * kConsumers) * 4;
    return p.ws_acc + ((row0 + o4 / D) * p.s_max + sp) * D + o4 % D;
  };
  float4 num[kOut];
  float M[kOut], den[kOut];
#pragma unroll
  for (int k = 0; k < kOut; ++k) {
    num[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    M[k] = -INFINITY;
    den[k] = 0.f;
  }

  for (int s0 = 0; s0 < nsplit; s0 += cap) {
    const int cnt = min(cap, nsplit - s0);
#pragma unroll
    for (int k = 0; k < kOut; ++k) {
      if (!valid(k)) continue;
      for (int sl = 0; sl < cnt; ++sl) cp_async16(rows + sl * kRow4 + tid + k * kConsumers, acc(k, s0 + sl));
    }
    for (int idx = tid; idx < G * cnt; idx += kConsumers) {
      const int i = idx / cnt, sl = idx - i * cnt;
      mlb[i * cap + sl] = __ldcg(ws_ml + (row0 + i) * p.s_max + s0 + sl);
    }
    cp_async_wait_all();
    named_barrier(1, kConsumers);  // the pairs, read by other threads
#pragma unroll
    for (int k = 0; k < kOut; ++k) {
      if (!valid(k)) continue;
      const float2* mk = mlb + head(k) * cap;
      float mc = M[k];
      for (int sl = 0; sl < cnt; ++sl) mc = fmaxf(mc, mk[sl].x);
      const float sc = fast_exp2(M[k] - mc);  // 0 on the first chunk
      num[k].x *= sc;
      num[k].y *= sc;
      num[k].z *= sc;
      num[k].w *= sc;
      den[k] *= sc;
      M[k] = mc;
      for (int sl = 0; sl < cnt; ++sl) {
        const float2 ml = mk[sl];
        const float4 x = rows[sl * kRow4 + tid + k * kConsumers];
        const float w = fast_exp2(ml.x - M[k]);
        num[k].x = fmaf(w, x.x, num[k].x);
        num[k].y = fmaf(w, x.y, num[k].y);
        num[k].z = fmaf(w, x.z, num[k].z);
        num[k].w = fmaf(w, x.w, num[k].w);
        den[k] = fmaf(w, ml.y, den[k]);
      }
    }
    named_barrier(1, kConsumers);  // the pairs are rewritten by the next chunk
  }
#pragma unroll
  for (int k = 0; k < kOut; ++k) {
    if (!valid(k)) continue;
    const int d = (tid + k * kConsumers) * 4 % D;
    OutT* dst = reinterpret_cast<OutT*>(p.out) + b * p.o_sb + (g * G + head(k)) * p.o_sh + d;
    store_out(dst + 0, num[k].x / den[k]);
    store_out(dst + 1, num[k].y / den[k]);
    store_out(dst + 2, num[k].z / den[k]);
    store_out(dst + 3, num[k].w / den[k]);
  }
}

// Minimum resident CTAs the register budget must allow: what shared memory
// allows at the default split length and ring depth (8 for G <= 4, 6 for G = 8).
template <int G>
constexpr int split_min_blocks() { return G <= 4 ? 8 : 6; }

template <int D, int G, typename OutT>
__global__ void __launch_bounds__(kThreads, split_min_blocks<G>()) paged_gqa_decode_split_kernel(const __grid_constant__ CUtensorMap tmk,
                                                                          const __grid_constant__ CUtensorMap tmv,
                                                                          const DecodeParams p) {
  constexpr int TILE_BYTES = kBlockSize * D * 2;
  constexpr int BOXES = D / kBoxDims;
  constexpr int KSTEPS = D / 16;  // 16-dim MMA steps (QK) = 16-dim m-tiles (PV)
  static_assert(D % kBoxDims == 0 && G >= 1 && G <= 8, "shape not built");

  // grid (KV head, sequence, split slot): the highest split index runs
  // first (split_work: splits are aligned to the end of the sequence).
  const int g = blockIdx.x, b = blockIdx.y, s = static_cast<int>(gridDim.z - 1 - blockIdx.z);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_launch_dependents();
  if (warp == kConsumerWarps) prefetch_first_stages<D>(&tmk, &tmv, p, b, g, s, p.nstage, lane);
  griddep_wait();  // every value used below is read after the previous grid in the stream is complete

  // The producer's block-table entries for this split are requested with the
  // length, not after it (a window that covers the split wherever the length
  // puts it; entries past the sequence are loaded but unused).
  TableWindow tw;
  if (warp == kConsumerWarps) {
    if (lane == 0) {  // the TMA descriptors, fetched while the length and table are read
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
    }
    tw.load(p, b, s, lane);
  }
  const int L = checked_length(p, b, s == 0 && g == 0 && threadIdx.x == 0);

  if (L == 0) {  // empty context: the output is defined as zero
    if (s == 0) {
      for (int o = threadIdx.x; o < G * D; o += kThreads) {
        const int i = o / D, d = o % D;
        store_out(reinterpret_cast<OutT*>(p.out) + b * p.o_sb + (g * G + i) * p.o_sh + d, 0.f);
      }
    }
    return;
  }
  const SplitWork sw = split_work(L, p.bps, s);
  const int nsplit = sw.nsplit;
  if (s >= nsplit) return;
  const int blk0 = sw.blk0;
  const int n = sw.n;  // KV blocks in this split (>= 1)
  const int nks = (n + kStageBlocks - 1) / kStageBlocks;  // stages per pass
  const int nstage = p.nstage;

  extern __shared__ __align__(128) unsigned char smem[];
  const SmemLayout lay = decode_layout(D, G, p.bps, nstage);
  const uint32_t sbase = smem_addr(smem);
  const uint32_t ring_s = (sbase + static_cast<uint32_t>(lay.ring)) & ~1023u;  // shared-space address
  unsigned char* ring = smem + (ring_s - sbase);
  float* red = reinterpret_cast<float*>(ring);  // consumer-warp merge, after the last stage
  float* logits = reinterpret_cast<float*>(smem + lay.logits);
  float* red_m = reinterpret_cast<float*>(smem + lay.red_ml);
  float* red_l = red_m + kConsumerWarps * G;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + lay.bars);
  uint64_t* empty = full + nstage;
  const int lrow = lay.lrow;

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
    if (tw.any_bad(blk0, n, p.NB, lane) && lane == 0) record_error(p.err, kDevErrBlockId);
    int slot = 0;
    uint32_t phase = 0;
    for (int i = 0; i < 2 * nks; ++i) {
      const bool is_v = i >= nks;
      const int j0 = (is_v ? i - nks : i) * kStageBlocks;
      int pb[kStageBlocks];
#pragma unroll
      for (int u = 0; u < kStageBlocks; ++u) {
        const int j = j0 + u;  // < bps + 1
        pb[u] = j < n ? tw.entry(blk0 + j) : -1;  // past the split: no tile
      }
      if (lane == 0) {
        if (i >= nstage) mbar_wait(empty + slot, phase ^ 1u, p.err);  // stage released
        uint32_t bytes = 0;
#pragma unroll
        for (int u = 0; u < kStageBlocks; ++u)
          if (static_cast<unsigned>(pb[u]) < static_cast<unsigned>(p.NB)) bytes += TILE_BYTES;
        if (bytes)
          mbar_arrive_expect_tx(full + slot, bytes);
        else
          mbar_arrive(full + slot);  // nothing to copy (bad ids are recorded above)
      }
      __syncwarp();
      // one (block, head) tile per lane: lane u copies block u
      if (lane < kStageBlocks) {
        int pbu = pb[0];
#pragma unroll
        for (int k = 1; k < kStageBlocks; ++k) pbu = lane == k ? pb[k] : pbu;
        if (static_cast<unsigned>(pbu) < static_cast<unsigned>(p.NB))
          tma_load_5d(ring + (slot * kStageBlocks + lane) * TILE_BYTES, is_v ? &tmv : &tmk, 0, 0, 0, g, pbu,
                      full + slot);
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
  const int tq = lane >> 2;     // MMA group id: a token (QK) / a dim (PV) row, and the head of B
  const int tr = lane & 3;      // MMA thread-in-group: a pair of columns
  const int t_base = blk0 * kBlockSize;

  // B operand of the QK product, q^T (k = dim, n = head), for all KSTEPS:
  // {q[tq][16ks + 2tr], +1} and {q[tq][16ks + 8 + 2tr], +1}; heads >= G are 0.
  // The optional q/k path runs at position L-1 (the new token's).
  const int pos = L - 1;
  const bool qk_path = p.q_norm_w != nullptr || p.k_norm_w != nullptr || p.rope != nullptr;
  const bool rope = p.rope != nullptr && pos < p.rope_rows;
  if (p.rope != nullptr && !rope && tid == 0 && s == 0 && g == 0) record_error(p.err, kDevErrPosition);
  const bool col_ok = PvCols<G>::valid(tq);  // column tq of the B operands holds a head
  uint32_t qb[KSTEPS][2];
  {
    const __nv_bfloat16* qrow =
        p.q + static_cast<int64_t>(b) * p.q_sb + static_cast<int64_t>(g * G + PvCols<G>::head(tq)) * p.q_sh;
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
      qb[ks][0] = col_ok ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * tr)) : 0u;
      qb[ks][1] = col_ok ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 8 + 2 * tr)) : 0u;
    }
    if (qk_path) {  // uniform across the CTA
      float x[KSTEPS][4];
#pragma unroll
      for (int ks = 0; ks < KSTEPS; ++ks) {
        x[ks][0] = bf16lo(qb[ks][0]);
        x[ks][1] = bf16hi(qb[ks][0]);
        x[ks][2] = bf16lo(qb[ks][1]);
        x[ks][3] = bf16hi(qb[ks][1]);
      }
      q_norm_rope<D>(x, tr, p, pos, rope);
#pragma unroll
      for (int ks = 0; ks < KSTEPS; ++ks) {
        qb[ks][0] = col_ok ? pack_bf16x2(x[ks][0], x[ks][1]) : 0u;
        qb[ks][1] = col_ok ? pack_bf16x2(x[ks][2], x[ks][3]) : 0u;
      }
    }
  }

  // Fused append: the split holding position L-1 patches that row of its last
  // block with this step's new K (pass 1) and V (pass 2), and stores it.
  const bool fused = p.k_new != nullptr && s == nsplit - 1;
  const int jl = n - 1, rl = (L - 1) % kBlockSize;  // block within the split, row
  __nv_bfloat16* kdst = nullptr;
  __nv_bfloat16* vdst = nullptr;
  if (fused) {
    const int pb = __ldg(p.block_tables + static_cast<int64_t>(b) * p.bt_sb + blk0 + jl);
    if (static_cast<unsigned>(pb) < static_cast<unsigned>(p.NB)) {  // a bad id is recorded by the producer
      kdst = p.k_cache_w + static_cast<int64_t>(pb) * p.kc_sblk + g * p.kc_sh + rl * D;
      vdst = p.v_cache_w + static_cast<int64_t>(pb) * p.vc_sblk + g * p.vc_sh + rl * D;
    }
  }

  int slot = 0;
  uint32_t phase = 0;

  // ---- pass 1: logits of every token of the split (log2 units), one tile per warp per stage
  for (int st = 0; st < nks; ++st) {
    mbar_wait(full + slot, phase, p.err);
    const int j = st * kStageBlocks + warp;  // block within the split
    if (j < n) {
      const uint32_t tile = ring_s + (slot * kStageBlocks + warp) * TILE_BYTES;
      if (fused && j == jl) {
        unsigned char* t = ring + (slot * kStageBlocks + warp) * TILE_BYTES;
        const __nv_bfloat16* src = p.k_new + static_cast<int64_t>(b) * p.kn_sb + g * p.kn_sh;
        if (qk_path)
          patch_new_k_row<D>(t, src, kdst, rl, lane, p, pos, rope);
        else
          patch_new_row<D>(t, src, kdst, rl, lane);
      }
      float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
      const int arow = (lane & 7) + ((lane >> 3) & 1) * 8;  // token row this lane addresses
      const int acol = lane >> 4;                           // +0 / +1 chunk
#pragma unroll
      for (int ks = 0; ks < KSTEPS; ++ks) {
        uint32_t a[4];
        ldsm_x4(swz(tile, arow, 2 * ks + acol), a);
        if (ks & 1)
          mma_16816_bf16(c1, a, qb[ks][0], qb[ks][1]);
        else
          mma_16816_bf16(c0, a, qb[ks][0], qb[ks][1]);
      }
      // c[0..1]: token tq, heads 2tr, 2tr+1; c[2..3]: token tq+8
      const int pos = t_base + j * kBlockSize;
      const bool v0 = pos + tq < L, v1 = pos + tq + 8 < L;
      const int h0 = 2 * tr, h1 = 2 * tr + 1;
      float* lg = logits + j * kBlockSize;
      if (h0 < G) {
        lg[h0 * lrow + tq] = v0 ? (c0[0] + c1[0]) * p.qk_scale_log2 : -INFINITY;
        lg[h0 * lrow + tq + 8] = v1 ? (c0[2] + c1[2]) * p.qk_scale_log2 : -INFINITY;
      }
      if (h1 < G) {
        lg[h1 * lrow + tq] = v0 ? (c0[1] + c1[1]) * p.qk_scale_log2 : -INFINITY;
        lg[h1 * lrow + tq + 8] = v1 ? (c0[3] + c1[3]) * p.qk_scale_log2 : -INFINITY;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + slot);
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
    for (int i = 0; i < G; ++i) {
      mx[i] = -INFINITY;
      for (int t = tid; t < ntok; t += kConsumers) mx[i] = fmaxf(mx[i], logits[i * lrow + t]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], off));
    }
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < G; ++i) red_m[warp * G + i] = mx[i];
    }
    named_barrier(1, kConsumers);
#pragma unroll
    for (int i = 0; i < G; ++i) {
      float m = red_m[i];
#pragma unroll
      for (int w = 1; w < kConsumerWarps; ++w) m = fmaxf(m, red_m[w * G + i]);
      float sum = 0.f;
      for (int t = tid; t < ntok; t += kConsumers) {
        const float e = fast_exp2(logits[i * lrow + t] - m);
        logits[i * lrow + t] = e;
        sum += e;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      if (lane == 0) red_l[warp * G + i] = sum;
    }
    named_barrier(1, kConsumers);
  }

  // ---- pass 2: O^T (dims x heads) += V^T P^T, one tile per warp per stage
  float o[KSTEPS][4];
#pragma unroll
  for (int mt = 0; mt < KSTEPS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;

  for (int st = 0; st < nks; ++st) {
    mbar_wait(full + slot, phase, p.err);
    const int j = st * kStageBlocks + warp;
    if (j < n) {
      const uint32_t tile = ring_s + (slot * kStageBlocks + warp) * TILE_BYTES;
      const int pos = t_base + j * kBlockSize;
      const int live = L - pos;  // >= 1 tokens of this block are in the sequence
      if (live < kBlockSize) {
        // the sequence ends inside this block: zero the V rows past its end
        // (they may hold anything, NaN included; P is 0 there but 0*NaN is NaN)
        unsigned char* trow = ring + (slot * kStageBlocks + warp) * TILE_BYTES;
        for (int idx = lane; idx < (kBlockSize - live) * BOXES * 8; idx += 32) {
          const int r = live + idx / (BOXES * 8), rest = idx % (BOXES * 8);
          *reinterpret_cast<uint4*>(trow + (rest >> 3) * kBoxBytes + r * 128 + (rest & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();  // before the TMA engine refills this stage
        __syncwarp();
      }
      if (fused && j == jl)
        patch_new_row<D>(ring + (slot * kStageBlocks + warp) * TILE_BYTES,
                         p.v_new + static_cast<int64_t>(b) * p.vn_sb + g * p.vn_sh, vdst, rl, lane);
      // B operand P^T (k = token, n = column tq): {p[2tr], +1}, {p[8 + 2tr], +1}
      // of the column's head, high or low part (PvCols)
      uint32_t bh0 = 0u, bh1 = 0u, bl0 = 0u, bl1 = 0u;
      if (col_ok) {
        const float* pr = logits + PvCols<G>::head(tq) * lrow + j * kBlockSize + 2 * tr;
        p_fragment<G>(tq, *reinterpret_cast<const float2*>(pr), *reinterpret_cast<const float2*>(pr + 8), bh0, bh1,
                      bl0, bl1);
      }
      const int arow = (lane & 7) + (lane >> 4) * 8;  // token row this lane addresses
      const int acol = (lane >> 3) & 1;               // +0 / +1 chunk
#pragma unroll
      for (int mt = 0; mt < KSTEPS; ++mt) {
        uint32_t a[4];
        ldsm_x4_trans(swz(tile, arow, 2 * mt + acol), a);
        mma_16816_bf16(o[mt], a, bh0, bh1);
        if (!PvCols<G>::kPacked) mma_16816_bf16(o[mt], a, bl0, bl1);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + slot);
    if (++slot == nstage) {
      slot = 0;
      phase ^= 1u;
    }
  }

  // ---- merge the consumer warps' partial O through shared memory (the ring
  // is free: every stage has been consumed)
  fold_low_columns<G>(o);
  named_barrier(1, kConsumers);
  {
    const int h0 = 2 * tr, h1 = 2 * tr + 1;
#pragma unroll
    for (int mt = 0; mt < KSTEPS; ++mt) {
      const int d0 = 16 * mt + tq, d1 = d0 + 8;
      if (h0 < G) {
        red[(warp * G + h0) * D + d0] = o[mt][0];
        red[(warp * G + h0) * D + d1] = o[mt][2];
      }
      if (h1 < G) {
        red[(warp * G + h1) * D + d0] = o[mt][1];
        red[(warp * G + h1) * D + d1] = o[mt][3];
      }
    }
  }
  named_barrier(1, kConsumers);

  for (int o4 = tid * 4; o4 < G * D; o4 += kConsumers * 4) {
    const int i = o4 / D, d = o4 % D;
    float4 t = *reinterpret_cast<const float4*>(red + i * D + d);
#pragma unroll
    for (int w = 1; w < kConsumerWarps; ++w) {
      const float4 x = *reinterpret_cast<const float4*>(red + (w * G + i) * D + d);
      t.x += x.x;
      t.y += x.y;
      t.z += x.z;
      t.w += x.w;
    }
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
  if (nsplit == 1) return;
  if (tid < G) {
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

  // ---- split reduce by the last CTA of (b, g) to arrive
  // Arrival: the barrier orders every consumer's partial stores before thread
  // 0's atomic, whose release half (cumulative over what the barrier ordered
  // before it) publishes them at GPU scope; in the last CTA, its acquire half
  // and the barrier order the other splits' partials before every thread's
  // reads -- the pattern of a grid-wide barrier.  One acquire-release atomic
  // in place of a fence, the atomic and a second fence: 0.5 us less on the
  // Qwen3-0.6B-shaped batch, whose time is mostly such round trips.
  named_barrier(1, kConsumers);
  int* counter = p.counters + static_cast<int64_t>(b) * p.Hkv + g;
  if (tid == 0) {
    int old;
    asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
    red_m[0] = __int_as_float(old == nsplit - 1 ? 1 : 0);
  }
  named_barrier(1, kConsumers);
  if (__float_as_int(red_m[0]) == 0) return;
  // the ring and the logits behind it are free now
  merge_splits<D, G, OutT>(p, b, g, nsplit, tid, red,
                           static_cast<int>((reinterpret_cast<unsigned char*>(red_m) - ring) / 4));
  if (tid == 0) *counter = 0;  // ready for the next call
}

// ---------------------------------------------------------------------------
// Single-pass variant: online softmax per block.
//
// The two-pass kernel above keeps every logit of a split in shared memory and
// stops streaming while it takes the split's softmax.  This one carries K and
// V of the same blocks in each stage (one block per consumer warp) and keeps,
// per warp and head, a running maximum and sum: per block it computes the
// 16 x G logits on the tensor cores, moves the maximum (rescaling that warp's
// O accumulators when it grows), and adds P V at once.  No logits buffer and
// no split-wide barrier: the ring streams without a pause and more of the
// shared memory holds data in flight.  The two warps' states are merged at
// the end (common maximum, rescaled sums), then the output or the split's
// partial is written exactly as above.
struct OnlineLayout {
  size_t ring, pscr, red_ml, bars, total;
};

// ring (1024-aligned; a stage is [K warp 0 | K warp 1 | V warp 0 | V warp 1],
// reused at the end for the consumer-warp merge) | per-warp P scratch
// [8 heads][16 tokens] fp32 | per-warp (max, sum) | mbarriers.
__host__ __device__ inline OnlineLayout online_layout(int D, int G, int nstage) {
  OnlineLayout l;
  size_t off = 1024;
  l.ring = off;
  const size_t ring = static_cast<size_t>(nstage) * kStageBlocks * 2 * kBlockSize * D * 2;
  const size_t red = static_cast<size_t>(kConsumerWarps) * G * D * 4;
  off += ring > red ? ring : red;
  l.pscr = off;
  off += static_cast<size_t>(kConsumerWarps) * 8 * kBlockSize * 4;
  l.red_ml = off;
  off += static_cast<size_t>(2) * kConsumerWarps * G * 4;
  off = (off + 15) & ~static_cast<size_t>(15);
  l.bars = off;
  off += static_cast<size_t>(2) * nstage * 8;
  l.total = off;
  return l;
}

template <int D, int G, typename OutT>
// Minimum resident CTAs stated for the single-pass kernel: 5, one more than
// its shared memory allows (4).  ptxas then keeps it at 128 registers and
// schedules it for that occupancy; measured against no minimum (the same
// register count): skewed batch 33.8 -> 32.9 us, 36-layer batch 70.5 -> 69.9 us
// per layer, Qwen3-4B-shaped 89.6 -> 89.5 us.  (A minimum of 4 let it take
// ~152 registers and cost the Qwen3-4B-shaped layer 15 %.)
__global__ void __launch_bounds__(kThreads, 5) paged_gqa_decode_online_kernel(const __grid_constant__ CUtensorMap tmk,
                                                                           const __grid_constant__ CUtensorMap tmv,
                                                                           const DecodeParams p) {
  constexpr int TILE_BYTES = kBlockSize * D * 2;
  constexpr int BOXES = D / kBoxDims;
  constexpr int KSTEPS = D / 16;
  static_assert(D % kBoxDims == 0 && G >= 1 && G <= 8, "shape not built");

  // grid (KV head, sequence, split slot): the highest split index runs
  // first (split_work: splits are aligned to the end of the sequence).
  const int g = blockIdx.x, b = blockIdx.y, s = static_cast<int>(gridDim.z - 1 - blockIdx.z);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_launch_dependents();
  if (warp == kConsumerWarps) prefetch_first_stages<D>(&tmk, &tmv, p, b, g, s, p.nstage, lane);
  griddep_wait();  // every value used below is read after the previous grid in the stream is complete

  // The producer's block-table entries for this split are requested with the
  // length, not after it (a window that covers the split wherever the length
  // puts it; entries past the sequence are loaded but unused).
  TableWindow tw;
  if (warp == kConsumerWarps) {
    if (lane == 0) {  // the TMA descriptors, fetched while the length and table are read
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
    }
    tw.load(p, b, s, lane);
  }
  const int L = checked_length(p, b, s == 0 && g == 0 && threadIdx.x == 0);

  if (L == 0) {  // empty context: the output is defined as zero
    if (s == 0) {
      for (int o = threadIdx.x; o < G * D; o += kThreads) {
        const int i = o / D, d = o % D;
        store_out(reinterpret_cast<OutT*>(p.out) + b * p.o_sb + (g * G + i) * p.o_sh + d, 0.f);
      }
    }
    return;
  }
  const SplitWork sw = split_work(L, p.bps, s);
  const int nsplit = sw.nsplit;
  if (s >= nsplit) return;
  const int blk0 = sw.blk0;
  const int n = sw.n;  // KV blocks in this split (>= 1)
  const int nst = (n + kStageBlocks - 1) / kStageBlocks;  // stages (K and V of 2 blocks each)
  const int nstage = p.nstage;

  extern __shared__ __align__(128) unsigned char smem[];
  const OnlineLayout lay = online_layout(D, G, nstage);
  const uint32_t sbase = smem_addr(smem);
  const uint32_t ring_s = (sbase + static_cast<uint32_t>(lay.ring)) & ~1023u;
  unsigned char* ring = smem + (ring_s - sbase);
  float* red = reinterpret_cast<float*>(ring);  // consumer-warp merge, after the last stage
  float* pscr = reinterpret_cast<float*>(smem + lay.pscr);
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
    if (tw.any_bad(blk0, n, p.NB, lane) && lane == 0) record_error(p.err, kDevErrBlockId);
    int slot = 0;
    uint32_t phase = 0;
    for (int st = 0; st < nst; ++st) {
      int pb[kStageBlocks];
#pragma unroll
      for (int u = 0; u < kStageBlocks; ++u) {
        const int j = st * kStageBlocks + u;  // < bps + 1
        pb[u] = j < n ? tw.entry(blk0 + j) : -1;  // past the split: no tile
      }
      if (lane == 0) {
        if (st >= nstage) mbar_wait(empty + slot, phase ^ 1u, p.err);  // stage released
        uint32_t bytes = 0;
#pragma unroll
        for (int u = 0; u < kStageBlocks; ++u)
          if (static_cast<unsigned>(pb[u]) < static_cast<unsigned>(p.NB)) bytes += 2 * TILE_BYTES;
        if (bytes)
          mbar_arrive_expect_tx(full + slot, bytes);
        else
          mbar_arrive(full + slot);  // nothing to copy (bad ids are recorded above)
      }
      __syncwarp();
      // one (block, head) tile per lane: lane 2 u + kv copies block u's K
      // (kv 0) or V (kv 1)
      if (lane < kStageBlocks * 2) {
        const int u = lane / 2, kv = lane % 2;
        int pbu = pb[0];
#pragma unroll
        for (int k = 1; k < kStageBlocks; ++k) pbu = u == k ? pb[k] : pbu;
        if (static_cast<unsigned>(pbu) < static_cast<unsigned>(p.NB))
          tma_load_5d(ring + (slot * 2 * kStageBlocks + kv * kStageBlocks + u) * TILE_BYTES, kv ? &tmv : &tmk, 0, 0,
                      0, g, pbu, full + slot);
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
  const int tq = lane >> 2;     // MMA group id: a token (QK) / a dim (PV) row, and the head of B
  const int tr = lane & 3;      // MMA thread-in-group: a pair of columns
  const int t_base = blk0 * kBlockSize;

  // B operand of QK^T, q^T (k = dim, n = head), for all KSTEPS; heads >= G are 0.
  // The optional q/k path runs at position L-1 (the new token's).
  const int pos = L - 1;
  const bool qk_path = p.q_norm_w != nullptr || p.k_norm_w != nullptr || p.rope != nullptr;
  const bool rope = p.rope != nullptr && pos < p.rope_rows;
  if (p.rope != nullptr && !rope && tid == 0 && s == 0 && g == 0) record_error(p.err, kDevErrPosition);
  const bool col_ok = PvCols<G>::valid(tq);  // column tq of the B operands holds a head
  uint32_t qb[KSTEPS][2];
  {
    const __nv_bfloat16* qrow =
        p.q + static_cast<int64_t>(b) * p.q_sb + static_cast<int64_t>(g * G + PvCols<G>::head(tq)) * p.q_sh;
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
      qb[ks][0] = col_ok ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * tr)) : 0u;
      qb[ks][1] = col_ok ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 8 + 2 * tr)) : 0u;
    }
    if (qk_path) {  // uniform across the CTA
      float x[KSTEPS][4];
#pragma unroll
      for (int ks = 0; ks < KSTEPS; ++ks) {
        x[ks][0] = bf16lo(qb[ks][0]);
        x[ks][1] = bf16hi(qb[ks][0]);
        x[ks][2] = bf16lo(qb[ks][1]);
        x[ks][3] = bf16hi(qb[ks][1]);
      }
      q_norm_rope<D>(x, tr, p, pos, rope);
#pragma unroll
      for (int ks = 0; ks < KSTEPS; ++ks) {
        qb[ks][0] = col_ok ? pack_bf16x2(x[ks][0], x[ks][1]) : 0u;
        qb[ks][1] = col_ok ? pack_bf16x2(x[ks][2], x[ks][3]) : 0u;
      }
    }
  }

  // Fused append: the split holding position L-1 patches that row of its last
  // block with this step's new K (before QK^T) and V (before P V), and stores it.
  const bool fused = p.k_new != nullptr && s == nsplit - 1;
  const int jl = n - 1, rl = (L - 1) % kBlockSize;  // block within the split, row
  __nv_bfloat16* kdst = nullptr;
  __nv_bfloat16* vdst = nullptr;
  if (fused) {
    const int pb = __ldg(p.block_tables + static_cast<int64_t>(b) * p.bt_sb + blk0 + jl);
    if (static_cast<unsigned>(pb) < static_cast<unsigned>(p.NB)) {  // a bad id is recorded by the producer
      kdst = p.k_cache_w + static_cast<int64_t>(pb) * p.kc_sblk + g * p.kc_sh + rl * D;
      vdst = p.v_cache_w + static_cast<int64_t>(pb) * p.vc_sblk + g * p.vc_sh + rl * D;
    }
  }

  // Running state of this warp for heads h0 = 2 tr, h1 = 2 tr + 1 (the S and
  // O accumulator columns this thread holds): maximum (log2 units) and this
  // lane's part of the sum; O^T (dims x heads) accumulators.
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[KSTEPS][4];
#pragma unroll
  for (int mt = 0; mt < KSTEPS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  float* psc = pscr + warp * 8 * kBlockSize;  // this warp's P^T scratch [head][token]

  int slot = 0;
  uint32_t phase = 0;
  for (int st = 0; st < nst; ++st) {
    mbar_wait(full + slot, phase, p.err);
    const int j = st * kStageBlocks + warp;  // block within the split
    if (j < n) {
      unsigned char* kt = ring + (slot * 2 * kStageBlocks + warp) * TILE_BYTES;
      unsigned char* vt = ring + (slot * 2 * kStageBlocks + kStageBlocks + warp) * TILE_BYTES;
      const uint32_t kt_s = ring_s + (slot * 2 * kStageBlocks + warp) * TILE_BYTES;
      const uint32_t vt_s = ring_s + (slot * 2 * kStageBlocks + kStageBlocks + warp) * TILE_BYTES;
      if (fused && j == jl) {
        const __nv_bfloat16* src = p.k_new + static_cast<int64_t>(b) * p.kn_sb + g * p.kn_sh;
        if (qk_path)
          patch_new_k_row<D>(kt, src, kdst, rl, lane, p, pos, rope);
        else
          patch_new_row<D>(kt, src, kdst, rl, lane);
      }
      // ---- S^T = K q^T: 16 tokens x 8 heads
      float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const int arow = (lane & 7) + ((lane >> 3) & 1) * 8;  // token row this lane addresses
        const int acol = lane >> 4;                           // +0 / +1 chunk
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks) {
          uint32_t a[4];
          ldsm_x4(swz(kt_s, arow, 2 * ks + acol), a);
          if (ks & 1)
            mma_16816_bf16(c1, a, qb[ks][0], qb[ks][1]);
          else
            mma_16816_bf16(c0, a, qb[ks][0], qb[ks][1]);
        }
      }
      const int tpos = t_base + j * kBlockSize;
      const bool v0 = tpos + tq < L, v1 = tpos + tq + 8 < L;
      const float s00 = v0 ? (c0[0] + c1[0]) * p.qk_scale_log2 : -INFINITY;  // token tq, head h0
      const float s01 = v0 ? (c0[1] + c1[1]) * p.qk_scale_log2 : -INFINITY;  // token tq, head h1
      const float s10 = v1 ? (c0[2] + c1[2]) * p.qk_scale_log2 : -INFINITY;  // token tq + 8, head h0
      const float s11 = v1 ? (c0[3] + c1[3]) * p.qk_scale_log2 : -INFINITY;  // token tq + 8, head h1
      // the block's maximum per head: over the 8 lanes sharing tr (every block
      // of the split holds at least one token of the sequence, so it is finite)
      float mt0 = fmaxf(s00, s10), mt1 = fmaxf(s01, s11);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mt0 = fmaxf(mt0, __shfl_xor_sync(0xffffffffu, mt0, off));
        mt1 = fmaxf(mt1, __shfl_xor_sync(0xffffffffu, mt1, off));
      }
      const float mn0 = fmaxf(m0, mt0), mn1 = fmaxf(m1, mt1);
      const float a0 = fast_exp2(m0 - mn0), a1 = fast_exp2(m1 - mn1);  // 0 on the first block
      m0 = mn0;
      m1 = mn1;
      const float p00 = fast_exp2(s00 - mn0), p01 = fast_exp2(s01 - mn1);
      const float p10 = fast_exp2(s10 - mn0), p11 = fast_exp2(s11 - mn1);
      l0 = fmaf(l0, a0, p00 + p10);
      l1 = fmaf(l1, a1, p01 + p11);
      if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
        for (int mt = 0; mt < KSTEPS; ++mt) {
          o[mt][0] *= a0;
          o[mt][1] *= a1;
          o[mt][2] *= a0;
          o[mt][3] *= a1;
        }
      }
      // P^T through the scratch: [head][token]
      psc[(2 * tr) * kBlockSize + tq] = p00;
      psc[(2 * tr + 1) * kBlockSize + tq] = p01;
      psc[(2 * tr) * kBlockSize + tq + 8] = p10;
      psc[(2 * tr + 1) * kBlockSize + tq + 8] = p11;
      const int live = L - tpos;  // >= 1 tokens of this block are in the sequence
      if (live < kBlockSize) {
        // the sequence ends inside this block: zero the V rows past its end
        // (they may hold anything, NaN included; P is 0 there but 0*NaN is NaN)
        for (int idx = lane; idx < (kBlockSize - live) * BOXES * 8; idx += 32) {
          const int r = live + idx / (BOXES * 8), rest = idx % (BOXES * 8);
          *reinterpret_cast<uint4*>(vt + (rest >> 3) * kBoxBytes + r * 128 + (rest & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();  // before the TMA engine refills this stage
      }
      __syncwarp();
      if (fused && j == jl)
        patch_new_row<D>(vt, p.v_new + static_cast<int64_t>(b) * p.vn_sb + g * p.vn_sh, vdst, rl, lane);
      // ---- O^T += V^T P^T, P as bf16 high + low parts (~16 significant
      // bits, whatever the output type): for G <= 4 in one MMA per 16 dims,
      // the low parts in the columns no head uses (PvCols), else two MMAs.
      // Column tq of the scratch holds the weights of its head (columns c
      // and c + 4 are equal when packed).
      uint32_t bh0 = 0u, bh1 = 0u, bl0 = 0u, bl1 = 0u;
      if (col_ok)
        p_fragment<G>(tq, *reinterpret_cast<const float2*>(psc + tq * kBlockSize + 2 * tr),
                      *reinterpret_cast<const float2*>(psc + tq * kBlockSize + 8 + 2 * tr), bh0, bh1, bl0, bl1);
      {
        const int arow = (lane & 7) + (lane >> 4) * 8;  // token row this lane addresses
        const int acol = (lane >> 3) & 1;               // +0 / +1 chunk
#pragma unroll
        for (int mt = 0; mt < KSTEPS; ++mt) {
          uint32_t a[4];
          ldsm_x4_trans(swz(vt_s, arow, 2 * mt + acol), a);
          mma_16816_bf16(o[mt], a, bh0, bh1);
          if (!PvCols<G>::kPacked) mma_16816_bf16(o[mt], a, bl0, bl1);
        }
      }
    }
    __syncwarp();  // the scratch is rewritten by the next block
    if (lane == 0) mbar_arrive(empty + slot);
    if (++slot == nstage) {
      slot = 0;
      phase ^= 1u;
    }
  }


  // ---- merge the two warps' states: per head, the common maximum M; each
  // warp's O and sum scaled by 2^(m_w - M) (0 for a warp that had no block)
  fold_low_columns<G>(o);
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  const int h0 = 2 * tr, h1 = 2 * tr + 1;
  named_barrier(1, kConsumers);  // both warps are done with the ring; it is reused below
  if (tq == 0) {
    if (h0 < G) red_m[warp * G + h0] = m0;
    if (h1 < G) red_m[warp * G + h1] = m1;
  }
  named_barrier(1, kConsumers);
  float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
  for (int w = 0; w < kConsumerWarps; ++w) {
    if (h0 < G) M0 = fmaxf(M0, red_m[w * G + h0]);
    if (h1 < G) M1 = fmaxf(M1, red_m[w * G + h1]);
  }
  const float f0 = h0 < G ? fast_exp2(m0 - M0) : 0.f, f1 = h1 < G ? fast_exp2(m1 - M1) : 0.f;
  if (tq == 0) {
    if (h0 < G) red_l[warp * G + h0] = l0 * f0;
    if (h1 < G) red_l[warp * G + h1] = l1 * f1;
  }
#pragma unroll
  for (int mt = 0; mt < KSTEPS; ++mt) {
    const int d0 = 16 * mt + tq, d1 = d0 + 8;
    if (h0 < G) {
      red[(warp * G + h0) * D + d0] = o[mt][0] * f0;
      red[(warp * G + h0) * D + d1] = o[mt][2] * f0;
    }
    if (h1 < G) {
      red[(warp * G + h1) * D + d0] = o[mt][1] * f1;
      red[(warp * G + h1) * D + d1] = o[mt][3] * f1;
    }
  }
  named_barrier(1, kConsumers);

  for (int o4 = tid * 4; o4 < G * D; o4 += kConsumers * 4) {
    const int i = o4 / D, d = o4 % D;
    float4 t = *reinterpret_cast<const float4*>(red + i * D + d);
#pragma unroll
    for (int w = 1; w < kConsumerWarps; ++w) {
      const float4 x = *reinterpret_cast<const float4*>(red + (w * G + i) * D + d);
      t.x += x.x;
      t.y += x.y;
      t.z += x.z;
      t.w += x.w;
    }
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
  if (nsplit == 1) return;
  if (tid < G) {
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

  // ---- split reduce by the last CTA of (b, g) to arrive
  // Arrival: the barrier orders every consumer's partial stores before thread
  // 0's atomic, whose release half (cumulative over what the barrier ordered
  // before it) publishes them at GPU scope; in the last CTA, its acquire half
  // and the barrier order the other splits' partials before every thread's
  // reads -- the pattern of a grid-wide barrier.  One acquire-release atomic
  // in place of a fence, the atomic and a second fence: 0.5 us less on the
  // Qwen3-0.6B-shaped batch, whose time is mostly such round trips.
  named_barrier(1, kConsumers);
  int* counter = p.counters + static_cast<int64_t>(b) * p.Hkv + g;
  if (tid == 0) {
    int old;
    asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
    red_m[0] = __int_as_float(old == nsplit - 1 ? 1 : 0);
  }
  named_barrier(1, kConsumers);
  if (__float_as_int(red_m[0]) == 0) return;
  // the ring and the P scratch behind it are free now
  merge_splits<D, G, OutT>(p, b, g, nsplit, tid, red,
                           static_cast<int>((reinterpret_cast<unsigned char*>(red_m) - ring) / 4));
  if (tid == 0) *counter = 0;  // ready for the next call
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
cudaError_t launch_typed(const DecodeParams& p, const CUtensorMap& tmk, const CUtensorMap& tmv,
                         cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(p.Hkv), static_cast<unsigned>(p.B), static_cast<unsigned>(p.s_max));
  if (p.online) {
    const size_t smem = online_layout(D, G, p.nstage).total;
    auto kernel = paged_gqa_decode_online_kernel<D, G, OutT>;
    static std::atomic<size_t> smem_set[64];  // one record per instantiation
    cudaError_t e = ensure_smem(kernel, smem, smem_set);
    if (e != cudaSuccess) return e;
    return launch_pdl(kernel, grid, dim3(kThreads), smem, stream, tmk, tmv, p);
  }
  const size_t smem = decode_layout(D, G, p.bps, p.nstage).total;
  auto split_kernel = paged_gqa_decode_split_kernel<D, G, OutT>;
  static std::atomic<size_t> smem_set[64];  // one record per instantiation
  cudaError_t e = ensure_smem(split_kernel, smem, smem_set);
  if (e != cudaSuccess) return e;
  return launch_pdl(split_kernel, grid, dim3(kThreads), smem, stream, tmk, tmv, p);
}

template <int D, typename OutT>
cudaError_t launch_g(const DecodeParams& p, const CUtensorMap& tmk, const CUtensorMap& tmv, int G,
                     cudaStream_t stream) {
  switch (G) {
    case 1: return launch_typed<D, 1, OutT>(p, tmk, tmv, stream);
    case 2: return launch_typed<D, 2, OutT>(p, tmk, tmv, stream);
    case 4: return launch_typed<D, 4, OutT>(p, tmk, tmv, stream);
    case 8: return launch_typed<D, 8, OutT>(p, tmk, tmv, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

size_t decode_smem_bytes(int D, int G, int bps, int nstage) {
  return decode_layout(D, G, bps, nstage).total;
}

cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& tmk, const CUtensorMap& tmv, int D, int G,
                          bool out_bf16, cudaStream_t stream) {
  if (p.B == 0) return cudaSuccess;
  if (D == 128) {
    return out_bf16 ? launch_g<128, __nv_bfloat16>(p, tmk, tmv, G, stream)
                    : launch_g<128, float>(p, tmk, tmv, G, stream);
  }
  if (D == 64) {
    return out_bf16 ? launch_g<64, __nv_bfloat16>(p, tmk, tmv, G, stream)
                    : launch_g<64, float>(p, tmk, tmv, G, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace forge
