// Shared device helpers and launch parameter blocks for the paged-KV kernels.
//
// Everything here is sm_103a inline PTX or plain CUDA: mbarrier-tracked bulk
// (TMA engine) copies from global to shared memory, bounded waits that give
// up with an error code instead of hanging, and the parameter structs that
// the C ABI layer fills in.
#pragma once

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
  float* ws_acc;   // [B*Hq, s_max, D] unnormalised split accumulators
  float* ws_ml;    // [B*Hq, s_max, 2] split (max, sum) in log2 units
  int B, Hq, Hkv, NB, MB;
  int bps;         // KV blocks per split
  int s_max;       // split slots per (b, h) in the workspace
  int nstage;      // shared-memory ring depth (pipeline stages)
  float qk_scale_log2;  // scale * log2(e): logits come out in log2 units
  int* err;
};

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
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
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

// Launchers (defined in append.cu / decode.cu).
cudaError_t launch_append(const AppendParams& p, cudaStream_t stream);
cudaError_t launch_decode(const DecodeParams& p, int D, int G, bool out_bf16, cudaStream_t stream);
size_t decode_smem_bytes(int D, int G, int bps, int nstage);

}  // namespace forge
