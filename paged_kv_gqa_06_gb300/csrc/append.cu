// Paged-KV append: scatter each sequence's new K/V token into its block slot.
//
// "Make the Engine Talk", 1.2: each decode pass adds the one new token of
// every sequence to the cache.  The cache is the paged block pool of the
// forge-engine README ("What it implements", KV cache row): the slot index
// slot = block * 16 + offset says where the token goes.
//
// One thread moves one 16-byte chunk (8 bf16) of one row of K or V; rows are
// D/8 chunks, so a warp writes whole 256-byte rows (D = 128) with 16-byte
// stores.  The copy is bit-exact.  A negative slot skips the row; a slot
// past the pool is skipped and recorded as kDevErrSlot.
#include "common.cuh"

namespace forge {
namespace {

__global__ void __launch_bounds__(256) paged_kv_append_kernel(const AppendParams p) {
  griddep_launch_dependents();
  griddep_wait();  // the previous grid's writes (e.g. of k_new / v_new) are complete
  const int chunks = p.D >> 3;
  const int64_t rows = static_cast<int64_t>(p.B) * p.Hkv;
  const int64_t total = 2 * rows * chunks;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(idx % chunks);
    int64_t r = idx / chunks;
    const int h = static_cast<int>(r % p.Hkv);
    r /= p.Hkv;
    const int b = static_cast<int>(r % p.B);
    const bool is_v = r >= p.B;
    const int64_t slot = p.slots[b];
    if (slot < 0) continue;
    if (slot >= static_cast<int64_t>(p.NB) * kBlockSize) {
      if (h == 0 && c == 0 && !is_v) record_error(p.err, kDevErrSlot);
      continue;
    }
    const int64_t blk = slot / kBlockSize;
    const int64_t off = slot % kBlockSize;
    const __nv_bfloat16* src =
        is_v ? p.v_new + b * p.vn_sb + h * p.vn_sh : p.k_new + b * p.kn_sb + h * p.kn_sh;
    __nv_bfloat16* dst = is_v ? p.v_cache + blk * p.vc_sblk + h * p.vc_sh
                              : p.k_cache + blk * p.kc_sblk + h * p.kc_sh;
    dst += off * p.D + c * 8;
    src += c * 8;
    *reinterpret_cast<uint4*>(dst) = __ldg(reinterpret_cast<const uint4*>(src));
  }
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream) {
  const int64_t total = 2ll * p.B * p.Hkv * (p.D / 8);
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  if (blocks > 65535) blocks = 65535;  // grid-stride loop covers the rest
  return launch_pdl(paged_kv_append_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream, p);
}

}  // namespace forge
