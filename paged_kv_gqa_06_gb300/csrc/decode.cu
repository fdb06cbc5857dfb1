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
//     table and streams each (block, head) K tile, then each V tile (16 x D
//     bf16, one contiguous run) into a ring of shared-memory slots with
//     single bulk copies on the TMA engine, tracked by mbarriers;
//   * warps 0-3 consume: 8 lanes per token, D/8 dims per lane.  Pass 1 forms
//     the G logits of every token of the split (fp32 FMA on bf16 widened
//     exactly, 3-step shuffle reduction) into shared memory; the split's max
//     and sum are taken over all of them at once (no running rescale); pass 2
//     accumulates p * V in registers;
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

struct SmemLayout {
  size_t ring, logits, red_acc, red_ml, bars, total;
};

__host__ __device__ inline SmemLayout decode_layout(int D, int G, int bps, int nstage) {
  SmemLayout l;
  size_t off = 0;
  l.ring = off;
  off += static_cast<size_t>(nstage) * kBlockSize * D * 2;
  l.logits = off;
  off += static_cast<size_t>(bps) * kBlockSize * G * 4;
  l.red_acc = off;
  off += static_cast<size_t>(kConsumerWarps) * G * D * 4;
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

template <int D, int G, typename OutT>
__global__ void __launch_bounds__(kThreads) paged_gqa_decode_split_kernel(const DecodeParams p) {
  constexpr int DPL = D / 8;   // dims per lane (8 lanes per token)
  constexpr int WPL = DPL / 2; // bf16 pairs per lane
  constexpr int VEC = DPL / 8; // 16-byte vectors per lane
  constexpr int TILE = kBlockSize * D;
  constexpr uint32_t kTileBytes = TILE * sizeof(__nv_bfloat16);
  static_assert(D % 64 == 0, "8 lanes x whole 16-byte vectors per token row");

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
  const int n = min(p.bps, nblk - blk0);  // KV blocks in this split (>= 1)
  const int nstage = p.nstage;

  extern __shared__ __align__(128) unsigned char smem[];
  const SmemLayout lay = decode_layout(D, G, p.bps, nstage);
  __nv_bfloat16* ring = reinterpret_cast<__nv_bfloat16*>(smem + lay.ring);
  float* logits = reinterpret_cast<float*>(smem + lay.logits);
  float* red_acc = reinterpret_cast<float*>(smem + lay.red_acc);
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
    for (int i = 0; i < 2 * n; ++i) {
      const bool is_v = i >= n;
      const int j = is_v ? i - n : i;
      const int pb = __shfl_sync(0xffffffffu, j < 32 ? e0 : e1, j & 31);
      if (lane == 0) {
        if (i >= nstage) mbar_wait(empty + slot, phase ^ 1u, p.err);  // slot released
        if (static_cast<unsigned>(pb) < static_cast<unsigned>(p.NB)) {
          const __nv_bfloat16* src =
              is_v ? vbase + static_cast<int64_t>(pb) * p.vc_sblk : kbase + static_cast<int64_t>(pb) * p.kc_sblk;
          mbar_arrive_expect_tx(full + slot, kTileBytes);
          bulk_copy_g2s(ring + slot * TILE, src, kTileBytes, full + slot);
        } else {
          mbar_arrive(full + slot);  // bad block id (recorded): release the slot without data
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
  const int tok = tid >> 3;     // token of the tile this thread reads
  const int sub = tid & 7;
  const int d0 = sub * DPL;
  const int t_base = blk0 * kBlockSize;

  float qf[G][DPL];
#pragma unroll
  for (int i = 0; i < G; ++i) {
    const uint4* src = reinterpret_cast<const uint4*>(p.q + static_cast<int64_t>(b) * p.q_sb +
                                                      static_cast<int64_t>(g * G + i) * p.q_sh + d0);
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
      const uint4 w4 = __ldg(src + v);
      const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        qf[i][8 * v + 2 * k] = bf16lo(w[k]) * p.qk_scale_log2;
        qf[i][8 * v + 2 * k + 1] = bf16hi(w[k]) * p.qk_scale_log2;
      }
    }
  }

  int slot = 0;
  uint32_t phase = 0;

  // ---- pass 1: logits of every token of the split (log2 units)
  for (int j = 0; j < n; ++j) {
    mbar_wait(full + slot, phase, p.err);
    uint32_t kw[WPL];
    const uint4* src = reinterpret_cast<const uint4*>(ring + slot * TILE + tok * D + d0);
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
      const uint4 x = src[v];
      kw[4 * v] = x.x;
      kw[4 * v + 1] = x.y;
      kw[4 * v + 2] = x.z;
      kw[4 * v + 3] = x.w;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + slot);

    float part[G];
#pragma unroll
    for (int i = 0; i < G; ++i) part[i] = 0.f;
#pragma unroll
    for (int w = 0; w < WPL; ++w) {
      const float k0 = bf16lo(kw[w]), k1 = bf16hi(kw[w]);
#pragma unroll
      for (int i = 0; i < G; ++i) {
        part[i] = fmaf(qf[i][2 * w], k0, part[i]);
        part[i] = fmaf(qf[i][2 * w + 1], k1, part[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < G; ++i) {
      part[i] += __shfl_xor_sync(0xffffffffu, part[i], 1);
      part[i] += __shfl_xor_sync(0xffffffffu, part[i], 2);
      part[i] += __shfl_xor_sync(0xffffffffu, part[i], 4);
    }
    if (sub == 0) {
      const bool valid = t_base + j * kBlockSize + tok < L;
      if (!valid) {
#pragma unroll
        for (int i = 0; i < G; ++i) part[i] = -INFINITY;
      }
      store_row<G>(logits + (j * kBlockSize + tok) * G, part);
    }
    if (++slot == nstage) {
      slot = 0;
      phase ^= 1u;
    }
  }
  named_barrier(1, kConsumers);

  // ---- softmax over the split: max, then p = 2^(s - max) in place, and sum
  const int ntok = n * kBlockSize;
  float m[G];
  {
    float mx[G];
#pragma unroll
    for (int i = 0; i < G; ++i) mx[i] = -INFINITY;
    for (int t = tid; t < ntok; t += kConsumers) {
      float v[G];
      load_row<G>(logits + t * G, v);
#pragma unroll
      for (int i = 0; i < G; ++i) mx[i] = fmaxf(mx[i], v[i]);
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
      float v[G];
      load_row<G>(logits + t * G, v);
#pragma unroll
      for (int i = 0; i < G; ++i) {
        v[i] = fast_exp2(v[i] - m[i]);
        sum[i] += v[i];
      }
      store_row<G>(logits + t * G, v);
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
  float acc[G][DPL];
#pragma unroll
  for (int i = 0; i < G; ++i)
#pragma unroll
    for (int k = 0; k < DPL; ++k) acc[i][k] = 0.f;

  for (int j = 0; j < n; ++j) {
    mbar_wait(full + slot, phase, p.err);
    uint32_t vw[WPL];
    const uint4* src = reinterpret_cast<const uint4*>(ring + slot * TILE + tok * D + d0);
#pragma unroll
    for (int v = 0; v < VEC; ++v) {
      const uint4 x = src[v];
      vw[4 * v] = x.x;
      vw[4 * v + 1] = x.y;
      vw[4 * v + 2] = x.z;
      vw[4 * v + 3] = x.w;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + slot);
    if (t_base + j * kBlockSize + tok < L) {
      float w[G];
      load_row<G>(logits + (j * kBlockSize + tok) * G, w);
#pragma unroll
      for (int ww = 0; ww < WPL; ++ww) {
        const float v0 = bf16lo(vw[ww]), v1 = bf16hi(vw[ww]);
#pragma unroll
        for (int i = 0; i < G; ++i) {
          acc[i][2 * ww] = fmaf(w[i], v0, acc[i][2 * ww]);
          acc[i][2 * ww + 1] = fmaf(w[i], v1, acc[i][2 * ww + 1]);
        }
      }
    }
    if (++slot == nstage) {
      slot = 0;
      phase ^= 1u;
    }
  }

  // ---- combine the 16 token groups: lanes 8 and 16 apart, then the 4 warps
#pragma unroll
  for (int i = 0; i < G; ++i)
#pragma unroll
    for (int k = 0; k < DPL; ++k) {
      acc[i][k] += __shfl_xor_sync(0xffffffffu, acc[i][k], 8);
      acc[i][k] += __shfl_xor_sync(0xffffffffu, acc[i][k], 16);
    }
  if (lane < 8) {
#pragma unroll
    for (int i = 0; i < G; ++i)
#pragma unroll
      for (int k = 0; k < DPL; k += 4)
        *reinterpret_cast<float4*>(red_acc + (warp * G + i) * D + d0 + k) =
            make_float4(acc[i][k], acc[i][k + 1], acc[i][k + 2], acc[i][k + 3]);
  }
  named_barrier(1, kConsumers);

  float l[G];
#pragma unroll
  for (int i = 0; i < G; ++i) {
    l[i] = red_l[i];
#pragma unroll
    for (int w = 1; w < kConsumerWarps; ++w) l[i] += red_l[w * G + i];
  }
#pragma unroll
  for (int i = 0; i < G; ++i) {
    const int h = g * G + i;
    for (int d = tid; d < D; d += kConsumers) {
      float v = red_acc[i * D + d];
#pragma unroll
      for (int w = 1; w < kConsumerWarps; ++w) v += red_acc[(w * G + i) * D + d];
      if (nsplit == 1) {
        store_out(reinterpret_cast<OutT*>(p.out) + b * p.o_sb + h * p.o_sh + d, v / l[i]);
      } else {
        p.ws_acc[((static_cast<int64_t>(b) * p.Hq + h) * p.s_max + s) * D + d] = v;
      }
    }
    if (nsplit > 1 && tid == i) {
      const int64_t r = (static_cast<int64_t>(b) * p.Hq + h) * p.s_max + s;
      p.ws_ml[2 * r] = m[i];
      p.ws_ml[2 * r + 1] = l[i];
    }
  }
}

// Merge the split partials of every (b, h) whose sequence has more than one
// split: with M = max_s m_s and w_s = 2^(m_s - M),
//   out = sum_s w_s acc_s / sum_s w_s l_s.
// One warp per (b, h); each lane owns D/32 consecutive dims.
template <int D, typename OutT>
__global__ void __launch_bounds__(128) paged_gqa_decode_reduce_kernel(const DecodeParams p) {
  constexpr int DPT = D / 32;
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
  for (int s = 0; s < nsplit; ++s) {
    const float w = fast_exp2(ml[2 * s] - M);
    if constexpr (DPT == 4) {
      const float4 x = *reinterpret_cast<const float4*>(a + static_cast<int64_t>(s) * D);
      acc[0] = fmaf(w, x.x, acc[0]);
      acc[1] = fmaf(w, x.y, acc[1]);
      acc[2] = fmaf(w, x.z, acc[2]);
      acc[3] = fmaf(w, x.w, acc[3]);
    } else {
      const float2 x = *reinterpret_cast<const float2*>(a + static_cast<int64_t>(s) * D);
      acc[0] = fmaf(w, x.x, acc[0]);
      acc[1] = fmaf(w, x.y, acc[1]);
    }
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
