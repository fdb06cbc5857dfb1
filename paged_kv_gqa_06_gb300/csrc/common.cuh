// Shared device helpers and launch parameter blocks for the paged-KV kernels.
//
// Everything here is sm_103a inline PTX or plain CUDA: mbarrier-tracked bulk
// (TMA engine) copies from global to shared memory, bounded waits that give
// up with an error code instead of hanging, and the parameter structs that
// the C ABI layer fills in.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the library does not link libcuda)
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace forge {

constexpr int kBlockSize = 16;  // tokens per KV block

// Device-side error codes (mirror FORGE_DEVERR_* in include/forge_paged.h).
constexpr int kDevErrBlockId = 1;
constexpr int kDevErrLength = 2;
constexpr int kDevErrSlot = 3;
constexpr int kDevErrTimeout = 4;
constexpr int kDevErrPosition = 5;
constexpr int kDevErrQuery = 6;

// A wait on a pipeline barrier gives up after this long (ns of %globaltimer).
// A copy of a few KiB completes in microseconds; reaching this means a bug,
// and the kernel records kDevErrTimeout and finishes instead of hanging.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct AppendParams {
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  int64_t kn_sb, kn_sh, vn_sb, vn_sh;   // element strides of k_new / v_new
  const int64_t* slots;
  __nv_bfloat16* k_cache;
  __nv_bfloat16* v_cache;
  int64_t kc_sblk, kc_sh, vc_sblk, vc_sh;  // element strides of the caches
  int B, Hkv, D, NB;
  int* err;
};

struct DecodeParams {
  const __nv_bfloat16* q;
  int64_t q_sb, q_sh;
  const __nv_bfloat16* k_cache;
  const __nv_bfloat16* v_cache;
  int64_t kc_sblk, kc_sh, vc_sblk, vc_sh;
  const int32_t* block_tables;
  int64_t bt_sb;
  const int32_t* context_lens;
  void* out;
  int64_t o_sb, o_sh;
  int* counters;   // [B*Hkv] split arrivals per (sequence, KV head); zero between calls
  float* ws_acc;   // [B*Hq, s_max, D] unnormalised split accumulators
  float* ws_ml;    // [B*Hq, s_max, 2] split (max, sum) in log2 units
  int B, Hq, Hkv, NB, MB;
  int bps;         // KV blocks per split
  int s_max;       // split slots per (b, h) in the workspace
  int nstage;      // shared-memory ring depth (pipeline stages)
  int online;      // 1: single-pass online-softmax kernel; 0: two-pass kernel
  float qk_scale_log2;  // scale * log2(e): logits come out in log2 units
  // Fused append (all null for a plain decode): the new K/V row of sequence
  // b, KV head g, written at position L_b - 1 of the cache before use.
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  int64_t kn_sb, kn_sh, vn_sb, vn_sh;
  __nv_bfloat16* k_cache_w;
  __nv_bfloat16* v_cache_w;
  // Optional q/k path of the fused call (all null = none): per-head RMSNorm
  // weights [D] and rotary cos/sin rows [rope_rows, D] (cos in [0, D/2),
  // sin in [D/2, D)), applied at position L_b - 1 before q and the new k
  // are used (and k is stored).
  const __nv_bfloat16* q_norm_w;
  const __nv_bfloat16* k_norm_w;
  float norm_eps;
  const float* rope;
  int rope_rows;
  int* err;
};

// Paged prefill: the query tokens of sequence b are rows query_start[b] ..
// query_start[b+1]-1 of q / out, at the last n_b positions of its L_b
// cached tokens.
struct PrefillParams {
  const __nv_bfloat16* q;
  int64_t q_st, q_sh;          // token, head strides (elements)
  const int32_t* block_tables;
  int64_t bt_sb;
  const int32_t* context_lens;
  const int32_t* query_start;  // [B + 1]
  void* out;
  int64_t o_st, o_sh;
  int B, Hq, Hkv, NB, MB, T;
  float qk_scale_log2;
  int* err;
  // Context chunks (tcgen05 kernel): a work item whose context spans more
  // than chunk_stages 128-token stages is split into end-aligned chunks of at
  // most chunk_stages stages, one CTA each; each writes its rows' partial
  // (O, m, l) and the last to arrive merges them.  chunk_stages = 0: no split.
  int chunk_stages, max_chunks;
  int* counters;               // [items * Hkv] arrival counters, zero between calls
  float* ws_o;                 // [items * max_chunks][rows][D] fp32 partial O
  float* ws_ml;                // [items * max_chunks][rows][2] fp32 (m, l)
};

// Programmatic dependent launch.  The decode and append kernels are
// launched with programmatic stream serialization: the next grid in the
// stream may be launched once every CTA of this one has called
// griddep_launch_dependents, and every kernel calls griddep_wait, which
// returns once the previous grid in the stream has completed and its memory
// is visible, before any memory access whose value it uses and before any
// write.  Only the launch, CTA start-up and (in the decode kernels) L2
// prefetches of the first K/V tiles overlap.  (Without the launch attribute
// both are no-ops.)
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch `kernel` with programmatic stream serialization allowed.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

__device__ __forceinline__ void record_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Make the barrier initialisations visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait until the barrier phase with this parity has completed.  Returns false
// (after recording kDevErrTimeout) if that takes longer than kWaitLimitNs.
// Once a wait has timed out anywhere, later waits give up at once, so a
// broken pipeline ends quickly instead of spending the limit at every wait.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  if (err && *reinterpret_cast<volatile int*>(err) == kDevErrTimeout) return false;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      record_error(err, kDevErrTimeout);
      return false;
    }
  }
  return true;
}

// One contiguous global -> shared copy on the TMA engine, completing `bytes`
// of transaction count on `bar`.  dst, src 16-byte aligned; bytes % 16 == 0.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// 16 bytes global -> shared, asynchronous, through L2 only (.cg: no L1 copy,
// so data other SMs wrote and made visible is read as it is in L2).  The
// copies a thread issued are complete, and visible to that thread, after its
// cp_async_wait_all.  dst and src 16-byte aligned.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// One tiled box of a 3-D tensor map into shared memory (as tma_load_4d).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
      : "memory");
}

// One tiled box of a 4-D tensor map (TMA engine) into shared memory,
// completing its bytes on `bar`.  c0 is the innermost coordinate; c0 times
// the element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_addr(bar))
      : "memory");
}

// Prefetch one tiled box of a 4-D tensor map into L2: no shared memory, no
// completion to track.  Coordinates outside the tensor fetch nothing; c0
// times the element size must be a multiple of 16 bytes, as for a load.
__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap* map, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}

// One tiled box of a 5-D tensor map into shared memory (as tma_load_4d).
__device__ __forceinline__ void tma_load_5d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            int c4, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(smem_addr(bar))
      : "memory");
}

// Prefetch one tiled box of a 5-D tensor map into L2 (as tma_prefetch_4d).
__device__ __forceinline__ void tma_prefetch_5d(const CUtensorMap* map, int c0, int c1, int c2, int c3, int c4) {
  asm volatile("cp.async.bulk.prefetch.tensor.5d.L2.global.tile [%0, {%1, %2, %3, %4, %5}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
               : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Four 8x8 b16 matrices from shared memory; lanes 8i..8i+7 give the row
// addresses of matrix i, register i receives it (row lane/4, cols 2(lane%4)+{0,1}).
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

// As ldsm_x4, each matrix transposed (register i holds rows 2(lane%4)+{0,1}, col lane/4).
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr)
               : "memory");
}

// d += A (16x16 bf16, row) * B (16x8 bf16, col), fp32 accumulate, one warp.
__device__ __forceinline__ void mma_16816_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Barrier among the first `nthreads` threads of the CTA (named barrier `id`).
__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// bf16 pair (low element in bits 0..15) -> two floats, exactly.
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) { return make_float2(bf16lo(w), bf16hi(w)); }

// d = a * b + c on both lanes of a float pair with one packed fp32 FMA
// (sm_100-family f32x2 instruction; each lane rounds like a scalar fmaf).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

// Round two floats to bf16 and pack them (x0 in the low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float x0, float x1) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// d = a + b on both lanes of a float pair with one packed fp32 add.
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Round two floats to bf16 (hi, packed low/high = x0/x1) and the residuals
// x - hi to bf16 (lo): hi + lo carries ~16 significant bits.  The residual
// is exact in fp32 (x and its bf16 rounding share the leading bits).
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  const float2 r = ffma2(make_float2(bf16lo(hi), bf16hi(hi)), make_float2(-1.f, -1.f), make_float2(x0, x1));
  const __nv_bfloat162 rl = __floats2bfloat162_rn(r.x, r.y);
  lo = *reinterpret_cast<const uint32_t*>(&rl);
}

// A (block, head) K or V tile of 16 tokens x D bf16 in shared memory, as the
// TMA engine writes it from the cache's tensor map: D/64 boxes of 16 rows x
// 128 bytes, each with the 128-byte swizzle.
constexpr int kBoxDims = 64;                          // dims per box: one 128-byte swizzle span
constexpr int kBoxBytes = kBlockSize * kBoxDims * 2;  // 2 KiB

// Shared-memory address of 16-byte chunk `chunk` (of D/8) in row `row` of
// such a tile: box = chunk / 8, and within a box the chunk index is XORed
// with the row index mod 8.
__device__ __forceinline__ uint32_t swz(uint32_t tile, int row, int chunk) {
  return tile + (chunk >> 3) * kBoxBytes + row * 128 + ((((chunk & 7) ^ (row & 7))) << 4);
}

// Launchers (defined in append.cu / decode.cu / prefill.cu).
cudaError_t launch_append(const AppendParams& p, cudaStream_t stream);
cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v, int D, int G,
                          bool out_bf16, cudaStream_t stream);
size_t decode_smem_bytes(int D, int G, int bps, int nstage);
cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v, int D, int G,
                           bool out_bf16, cudaStream_t stream);
// The same prefill on the 5th-generation tensor cores; tmap_q is a 3-D map
// over q [T, Hq, D] with boxes of 64 dims x G heads x (128 / G) tokens.
cudaError_t launch_prefill_tc(const PrefillParams& p, const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                              const CUtensorMap& tmap_v, int D, int G, bool out_bf16, cudaStream_t stream);
// Its work items (query-tile pairs) for T query tokens over B sequences at
// group size G, an upper bound on the sequences' own counts; the grid has
// items * max(1, max_chunks) * Hkv CTAs.
int64_t prefill_tc_items(int64_t T, int64_t B, int G);
// The partial rows of one (item, KV head, chunk): two query tiles of 128.
constexpr int kPrefillChunkRows = 256;

}  // namespace forge
