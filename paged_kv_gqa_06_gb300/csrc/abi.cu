// C ABI of libforge_paged.so (declared in include/forge_paged.h).
//
// Host side only: argument validation, split planning from host-known shapes
// (no device reads, so calls stay asynchronous and capturable), the split
// workspace cache, the device error word, and the kernel launches.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <utility>

#include <cudaTypedefs.h>  // PFN_cuTensorMapEncodeTiled

#include "../../include/forge_paged.h"
#include "common.cuh"

namespace {

using forge::kBlockSize;

// Device error word: the first device-side precondition violation since the
// last forge_paged_get_device_error call.
__device__ int g_device_error;

constexpr int kMaxDevices = 64;
constexpr int kDefaultSplitTokens = 512;     // longest automatic split of the two-pass kernel
constexpr int kOnlineDeepRingTokens = 512;   // single-pass ring: 3 stages on splits from here up, 2 below
constexpr int kMaxSplitTokens = 1024;  // producer lanes hold <= 64 table entries
constexpr int kMinSplitTokens = 16;

std::mutex g_mu;
int* g_err_ptr[kMaxDevices];
int g_num_sms[kMaxDevices];

// Split workspace owned by the library, one per (device, stream).  Its own
// mutex is held from the lookup until the kernel that uses it is enqueued, so
// a call that grows it (and releases the old buffer in stream order) never
// runs between another call's lookup and launch on the same stream.
struct StreamScratch {
  std::mutex mu;
  void* ptr = nullptr;
  size_t bytes = 0;
};
std::map<std::pair<int, cudaStream_t>, std::unique_ptr<StreamScratch>> g_workspaces;  // guarded by g_mu

int current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices) return FORGE_ERR_CUDA;
  return FORGE_OK;
}

// Address of this device's error word (looked up once per device) and its SM count.
int device_state(int dev, int** err, int* sms) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return FORGE_ERR_CUDA;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return FORGE_ERR_CUDA;
    g_num_sms[dev] = n;
    g_err_ptr[dev] = static_cast<int*>(p);
  }
  *err = g_err_ptr[dev];
  *sms = g_num_sms[dev];
  return FORGE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_tensor(const forge_tensor* t, int dtype, int ndim) {
  if (!t) return FORGE_ERR_NULL;
  if (t->dtype != dtype) return FORGE_ERR_DTYPE;
  if (t->ndim != ndim) return FORGE_ERR_SHAPE;
  for (int i = 0; i < ndim; ++i)
    if (t->shape[i] < 0) return FORGE_ERR_SHAPE;
  return FORGE_OK;
}

int64_t numel(const forge_tensor* t) {
  int64_t n = 1;
  for (int i = 0; i < t->ndim; ++i) n *= t->shape[i];
  return n;
}

// bf16 tensor read/written in 16-byte vectors along its last dim: innermost
// stride 1, other strides multiples of 8 elements, data 16-byte aligned.
int check_vec16(const forge_tensor* t, int elem_bytes) {
  if (numel(t) == 0) return FORGE_OK;
  if (!t->data) return FORGE_ERR_NULL;
  if (t->stride[t->ndim - 1] != 1) return FORGE_ERR_SHAPE;
  const int64_t per16 = 16 / elem_bytes;
  for (int i = 0; i < t->ndim - 1; ++i)
    if (t->stride[i] % per16 != 0) return FORGE_ERR_ALIGN;
  if (!aligned16(t->data)) return FORGE_ERR_ALIGN;
  return FORGE_OK;
}

// [NB, Hkv, BS, D] bf16 cache: each (block, head) tile contiguous.
int check_cache(const forge_tensor* c) {
  int rc = check_tensor(c, FORGE_BF16, 4);
  if (rc) return rc;
  if (c->shape[2] != kBlockSize) return FORGE_ERR_UNSUPPORTED;
  if (numel(c) == 0) return FORGE_OK;
  if (c->stride[3] != 1 || c->stride[2] != c->shape[3]) return FORGE_ERR_SHAPE;
  return check_vec16(c, 2);
}

#define FORGE_TRY(expr)      \
  do {                       \
    int _rc = (expr);        \
    if (_rc != FORGE_OK) return _rc; \
  } while (0)

struct DecodePlan {
  forge::DecodeParams p;
  int D, G;
  bool out_bf16;
  size_t ws_bytes;
  const forge_tensor* k_cache;
  const forge_tensor* v_cache;
};

// cuTensorMapEncodeTiled from the driver, looked up through the runtime so
// that the library does not link libcuda.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      f = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// Tensor map over a [NB, Hkv, 16, D] bf16 cache, dims listed innermost first
// (D, token, head, block), boxes of 64 dims x 16 tokens (128-byte rows) with
// the 128-byte swizzle the kernels' shared-memory addressing expects.
int encode_cache_map(const forge_tensor* c, CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return FORGE_ERR_CUDA;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(c->shape[3]), static_cast<cuuint64_t>(kBlockSize),
                              static_cast<cuuint64_t>(c->shape[1]),
                              static_cast<cuuint64_t>(c->shape[0] > 0 ? c->shape[0] : 1)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(c->stride[2]) * 2, static_cast<cuuint64_t>(c->stride[1]) * 2,
                                 static_cast<cuuint64_t>(c->stride[0]) * 2};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(kBlockSize), 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  void* base = c->data;
  static unsigned char dummy[16] __attribute__((aligned(16)));
  if (!base) base = dummy;  // empty pool: the map is never used
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, base, dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FORGE_OK : FORGE_ERR_UNSUPPORTED;
}

// The same cache as a 5-D tensor map whose box is a whole (block, head) tile:
// dims innermost first (64 dims, token, 64-dim half, head, block), box
// 64 x 16 x D/64.  It lands as D/64 swizzled 2 KB sub-tiles of 16 rows x
// 128 bytes, one per half, the layout two boxes of the 4-D map give, in one
// copy instead of D/64.
int encode_cache_tile_map(const forge_tensor* c, CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return FORGE_ERR_CUDA;
  const cuuint64_t dims[5] = {64, static_cast<cuuint64_t>(kBlockSize), static_cast<cuuint64_t>(c->shape[3] / 64),
                              static_cast<cuuint64_t>(c->shape[1]),
                              static_cast<cuuint64_t>(c->shape[0] > 0 ? c->shape[0] : 1)};
  const cuuint64_t strides[4] = {static_cast<cuuint64_t>(c->stride[2]) * 2, 128,
                                 static_cast<cuuint64_t>(c->stride[1]) * 2, static_cast<cuuint64_t>(c->stride[0]) * 2};
  const cuuint32_t box[5] = {64, static_cast<cuuint32_t>(kBlockSize), static_cast<cuuint32_t>(c->shape[3] / 64), 1, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  void* base = c->data;
  static unsigned char dummy[16] __attribute__((aligned(16)));
  if (!base) base = dummy;  // empty pool: the map is never used
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, base, dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FORGE_OK : FORGE_ERR_UNSUPPORTED;
}

// Tensor map over the prefill's q [T, Hq, D] bf16, dims innermost first
// (D, head, token), boxes of 64 dims x G heads x 128/G tokens: one box is the
// 128 K-major rows (token-major, head-minor) of the tcgen05 kernel's Q tile,
// with the 128-byte swizzle.  Rows past T read as zeros.
int encode_q_map(const forge_tensor* q, int G, CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return FORGE_ERR_CUDA;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(q->shape[2]), static_cast<cuuint64_t>(q->shape[1]),
                              static_cast<cuuint64_t>(q->shape[0])};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(q->stride[1]) * 2, static_cast<cuuint64_t>(q->stride[0]) * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(128 / G)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q->data, dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FORGE_OK : FORGE_ERR_UNSUPPORTED;
}

// Which prefill kernel: the tcgen05 one unless FORGE_PREFILL_KERNEL=mma
// selects the mma.sync one (kept for comparison).
bool prefill_use_mma_sync() {
  const char* e = std::getenv("FORGE_PREFILL_KERNEL");
  return e && std::strcmp(e, "mma") == 0;
}

// Decode kernel forced by FORGE_DECODE_KERNEL ("online" or "two_pass"), read
// at every call; 0 when unset (the plan chooses).
int decode_kernel_forced() {
  const char* e = std::getenv("FORGE_DECODE_KERNEL");
  if (!e) return 0;
  if (std::strcmp(e, "online") == 0) return 2;
  if (std::strcmp(e, "two_pass") == 0) return 1;
  return 0;
}

// Split length (KV blocks) and decode kernel of a call.
//
// Automatic length: the longest split, from 1024 tokens halving down to 64,
// whose upper bound on CTAs (every sequence as long as its table row) gives
// ~4 CTAs per SM.  Shorter splits than that add more merge work than
// parallelism (measured: Qwen3-0.6B-shaped batch of 8, 12.8 us at 128-token
// splits against 16.0 us at 64).
//
// Kernel: the single-pass online-softmax kernel at every split length (its
// shared memory is all K/V ring, so more bytes are in flight per SM).  On
// short splits its ring is 2 stages deep, which lets a fifth CTA onto each SM
// (nstage_for).  Measured on GB300, decode of one layer: Qwen3-4B-shaped
// batch of 32, 93.6 us single-pass at 1024 tokens against 97.9 us two-pass at
// 512; Qwen3-0.6B-shaped batch of 8, 10.97 us single-pass at 128 tokens with
// 2 stages against 11.72 us two-pass.  FORGE_DECODE_KERNEL=two_pass selects
// the two-pass kernel.
int split_blocks_for(int split_tokens, int B, int Hkv, int MB, int num_sms, int* online) {
  int bps = kMaxSplitTokens / kBlockSize;
  if (split_tokens > 0) {
    bps = split_tokens / kBlockSize;
  } else {
    const int64_t want = 4ll * (num_sms > 0 ? num_sms : 148);
    while (bps > 4) {
      const int64_t ctas = static_cast<int64_t>(B) * Hkv * ((MB + bps - 1) / bps);
      if (ctas >= want) break;
      bps /= 2;
    }
  }
  const int forced = decode_kernel_forced();
  *online = forced ? (forced == 2) : 1;  // the two-pass kernel only when FORGE_DECODE_KERNEL asks
  if (split_tokens == 0 && !*online) bps = std::min(bps, kDefaultSplitTokens / kBlockSize);
  return bps;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Split workspace: a fixed prefix of kCounterSlots int32 arrival counters
// (one per (sequence, KV head), so B * Hkv <= kCounterSlots) | [B*Hq, s_max,
// D] fp32 accumulators | [B*Hq, s_max, 2] fp32 (max, sum).  The prefix has
// the same size for every shape, so no call's data ever lands on counters:
// once zeroed, the counters stay zero between calls (each call returns the
// ones it used to zero), whatever shapes share the workspace.
constexpr int64_t kCounterSlots = 65536;
constexpr size_t kCounterBytes = kCounterSlots * 4;
// Prefill context chunks: at most this many 128-token stages per fp32
// accumulation, and at most this much scratch for the chunks' partial rows.
constexpr int64_t kPrefillChunkStages = 32;
constexpr size_t kPrefillScratchCap = size_t(1) << 30;

size_t workspace_bytes_for(int64_t B, int64_t Hq, int64_t D, int64_t s_max) {
  if (s_max <= 1) return 0;
  const size_t acc = static_cast<size_t>(B * Hq * s_max * D) * 4;
  const size_t ml = static_cast<size_t>(B * Hq * s_max * 2) * 4;
  return kCounterBytes + round256(acc) + ml;
}

// Ring depth, unless FORGE_PAGED_NSTAGE sets one for both kernels.
// Single-pass kernel: 3 stages on splits of 512 tokens or more (Qwen3-4B-shaped
// batch at 1024: 94.2 us, against 96.1 and 99.6 at 2 and 4 stages); 2 on
// shorter splits, which the plan gives only to small problems: the smaller
// ring lets a fifth CTA onto each SM, so the grid runs in one wave
// (Qwen3-0.6B-shaped batch of 8 at 128-token splits: 10.97 us, against 13.95
// at 3 stages and 11.72 for the two-pass kernel).  Two-pass kernel (when
// forced): 3 on splits of up to 256 tokens (its logits buffer is small there,
// so the third stage costs no occupancy) and 2 above (Qwen3-4B-shaped batch
// at 512: 97.9 against 100.5 us).
int nstage_for(bool online, int bps) {
  static int v = [] {
    const char* e = std::getenv("FORGE_PAGED_NSTAGE");
    int n = e ? std::atoi(e) : 0;
    return (n >= 2 && n <= 16) ? n : 0;
  }();
  if (v) return v;
  if (online) return bps * kBlockSize >= kOnlineDeepRingTokens ? 3 : 2;
  return bps * kBlockSize <= 256 ? 3 : 2;
}

int plan_decode(const forge_tensor* q, const forge_tensor* k_cache, const forge_tensor* v_cache,
                const forge_tensor* block_tables, const forge_tensor* context_lens, float scale,
                forge_tensor* out, int split_tokens, int num_sms, DecodePlan* plan) {
  FORGE_TRY(check_tensor(q, FORGE_BF16, 3));
  FORGE_TRY(check_cache(k_cache));
  FORGE_TRY(check_cache(v_cache));
  FORGE_TRY(check_tensor(block_tables, FORGE_I32, 2));
  FORGE_TRY(check_tensor(context_lens, FORGE_I32, 1));
  if (!out) return FORGE_ERR_NULL;
  if (out->dtype != FORGE_BF16 && out->dtype != FORGE_F32) return FORGE_ERR_DTYPE;
  if (out->ndim != 3) return FORGE_ERR_SHAPE;

  const int64_t B = q->shape[0], Hq = q->shape[1], D = q->shape[2];
  const int64_t NB = k_cache->shape[0], Hkv = k_cache->shape[1];
  const int64_t MB = block_tables->shape[1];
  for (int i = 0; i < 4; ++i)
    if (v_cache->shape[i] != k_cache->shape[i]) return FORGE_ERR_SHAPE;
  if (k_cache->shape[3] != D) return FORGE_ERR_SHAPE;
  if (out->shape[0] != B || out->shape[1] != Hq || out->shape[2] != D) return FORGE_ERR_SHAPE;
  if (block_tables->shape[0] != B || context_lens->shape[0] != B) return FORGE_ERR_SHAPE;
  if (B > 65535 || Hkv > 65535 || NB > INT32_MAX || MB > (INT32_MAX / kBlockSize)) return FORGE_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return FORGE_ERR_UNSUPPORTED;
  if (Hkv <= 0 || Hq <= 0 || Hq % Hkv != 0) return (Hkv <= 0 || Hq <= 0) ? FORGE_ERR_SHAPE : FORGE_ERR_UNSUPPORTED;
  const int64_t G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return FORGE_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return FORGE_ERR_VALUE;
  if (split_tokens != 0 &&
      (split_tokens < kMinSplitTokens || split_tokens > kMaxSplitTokens || split_tokens % kBlockSize != 0))
    return FORGE_ERR_VALUE;

  std::memset(plan, 0, sizeof(*plan));
  plan->k_cache = k_cache;
  plan->v_cache = v_cache;
  plan->D = static_cast<int>(D);
  plan->G = static_cast<int>(G);
  plan->out_bf16 = out->dtype == FORGE_BF16;
  if (B == 0) return FORGE_OK;

  FORGE_TRY(check_vec16(q, 2));
  FORGE_TRY(check_vec16(out, out->dtype == FORGE_BF16 ? 2 : 4));
  if (!block_tables->data || !context_lens->data) return FORGE_ERR_NULL;
  if (block_tables->stride[1] != 1 || context_lens->stride[0] != 1) return FORGE_ERR_SHAPE;
  if (NB > 0 && (!k_cache->data || !v_cache->data)) return FORGE_ERR_NULL;

  forge::DecodeParams& p = plan->p;
  p.q = static_cast<const __nv_bfloat16*>(q->data);
  p.q_sb = q->stride[0];
  p.q_sh = q->stride[1];
  p.k_cache = static_cast<const __nv_bfloat16*>(k_cache->data);
  p.v_cache = static_cast<const __nv_bfloat16*>(v_cache->data);
  p.kc_sblk = k_cache->stride[0];
  p.kc_sh = k_cache->stride[1];
  p.vc_sblk = v_cache->stride[0];
  p.vc_sh = v_cache->stride[1];
  p.block_tables = static_cast<const int32_t*>(block_tables->data);
  p.bt_sb = block_tables->stride[0];
  p.context_lens = static_cast<const int32_t*>(context_lens->data);
  p.out = out->data;
  p.o_sb = out->stride[0];
  p.o_sh = out->stride[1];
  p.B = static_cast<int>(B);
  p.Hq = static_cast<int>(Hq);
  p.Hkv = static_cast<int>(Hkv);
  p.NB = static_cast<int>(NB);
  p.MB = static_cast<int>(MB);
  p.bps = split_blocks_for(split_tokens, p.B, p.Hkv, p.MB, num_sms, &p.online);
  p.s_max = MB > 0 ? static_cast<int>((MB + p.bps - 1) / p.bps) : 1;
  if (p.s_max > 65535) return FORGE_ERR_UNSUPPORTED;  // grid z limit
  p.nstage = nstage_for(p.online != 0, p.bps);
  p.qk_scale_log2 = scale * 1.4426950408889634f;
  plan->ws_bytes = workspace_bytes_for(B, Hq, D, p.s_max);
  if (plan->ws_bytes > 0 && B * Hkv > kCounterSlots) return FORGE_ERR_UNSUPPORTED;
  return FORGE_OK;
}

void attach_workspace(DecodePlan* plan, void* ws) {
  forge::DecodeParams& p = plan->p;
  if (plan->ws_bytes == 0) {
    p.counters = nullptr;
    p.ws_acc = nullptr;
    p.ws_ml = nullptr;
    return;
  }
  char* base = static_cast<char*>(ws);
  const size_t acc = round256(static_cast<size_t>(p.B) * p.Hq * p.s_max * plan->D * 4);
  p.counters = reinterpret_cast<int*>(base);
  p.ws_acc = reinterpret_cast<float*>(base + kCounterBytes);
  p.ws_ml = reinterpret_cast<float*>(base + kCounterBytes + acc);
}

int launch_plan(DecodePlan* plan, cudaStream_t stream) {
  CUtensorMap tmk, tmv;
  FORGE_TRY(encode_cache_tile_map(plan->k_cache, &tmk));
  FORGE_TRY(encode_cache_tile_map(plan->v_cache, &tmv));
  if (forge::launch_decode(plan->p, tmk, tmv, plan->D, plan->G, plan->out_bf16, stream) != cudaSuccess)
    return FORGE_ERR_CUDA;
  return FORGE_OK;
}

// Library-owned workspace for (device, stream), grown on demand with
// stream-ordered allocation: the new buffer is allocated and zero-filled on
// `stream` (the split arrival counters start at zero; kernels return them to
// zero), and the old one is released with cudaFreeAsync on the same stream,
// after the work already queued there.  No host synchronisation.  Growth is
// refused while `stream` is being captured (the buffer would belong to the
// graph).  On success `hold` owns the scratch's lock: the caller keeps it
// until its kernel is enqueued.
int cached_workspace(int dev, cudaStream_t stream, size_t bytes, void** out, std::unique_lock<std::mutex>* hold) {
  StreamScratch* sc = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    auto& slot = g_workspaces[{dev, stream}];
    if (!slot) slot.reset(new StreamScratch);
    sc = slot.get();  // never removed, so the pointer stays valid
  }
  std::unique_lock<std::mutex> lock(sc->mu);
  if (sc->bytes < bytes) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return FORGE_ERR_CUDA;
    if (cap != cudaStreamCaptureStatusNone) return FORGE_ERR_WORKSPACE;
    void* p = nullptr;
    if (cudaMallocAsync(&p, bytes, stream) != cudaSuccess) return FORGE_ERR_CUDA;
    if (cudaMemsetAsync(p, 0, bytes, stream) != cudaSuccess) {
      cudaFreeAsync(p, stream);
      return FORGE_ERR_CUDA;
    }
    if (sc->ptr && cudaFreeAsync(sc->ptr, stream) != cudaSuccess) {
      cudaFreeAsync(p, stream);
      return FORGE_ERR_CUDA;
    }
    sc->ptr = p;
    sc->bytes = bytes;
  }
  *out = sc->ptr;
  *hold = std::move(lock);
  return FORGE_OK;
}

}  // namespace

extern "C" {

int forge_paged_kv_append(const forge_tensor* k_new, const forge_tensor* v_new,
                          const forge_tensor* slot_mapping, forge_tensor* k_cache,
                          forge_tensor* v_cache, void* stream) {
  FORGE_TRY(check_tensor(k_new, FORGE_BF16, 3));
  FORGE_TRY(check_tensor(v_new, FORGE_BF16, 3));
  FORGE_TRY(check_tensor(slot_mapping, FORGE_I64, 1));
  FORGE_TRY(check_cache(k_cache));
  FORGE_TRY(check_cache(v_cache));
  const int64_t B = k_new->shape[0], Hkv = k_new->shape[1], D = k_new->shape[2];
  for (int i = 0; i < 3; ++i)
    if (v_new->shape[i] != k_new->shape[i]) return FORGE_ERR_SHAPE;
  for (int i = 0; i < 4; ++i)
    if (v_cache->shape[i] != k_cache->shape[i]) return FORGE_ERR_SHAPE;
  if (slot_mapping->shape[0] != B || k_cache->shape[1] != Hkv || k_cache->shape[3] != D) return FORGE_ERR_SHAPE;
  if (D % 8 != 0) return FORGE_ERR_UNSUPPORTED;
  if (B > INT32_MAX || Hkv > INT32_MAX || k_cache->shape[0] > INT32_MAX) return FORGE_ERR_UNSUPPORTED;
  if (B == 0 || Hkv == 0 || D == 0) return FORGE_OK;
  FORGE_TRY(check_vec16(k_new, 2));
  FORGE_TRY(check_vec16(v_new, 2));
  if (!slot_mapping->data) return FORGE_ERR_NULL;
  if (slot_mapping->stride[0] != 1) return FORGE_ERR_SHAPE;
  if (k_cache->shape[0] > 0 && (!k_cache->data || !v_cache->data)) return FORGE_ERR_NULL;

  int dev = 0, sms = 0;
  int* err = nullptr;
  FORGE_TRY(current_device(&dev));
  FORGE_TRY(device_state(dev, &err, &sms));

  forge::AppendParams p;
  p.k_new = static_cast<const __nv_bfloat16*>(k_new->data);
  p.v_new = static_cast<const __nv_bfloat16*>(v_new->data);
  p.kn_sb = k_new->stride[0];
  p.kn_sh = k_new->stride[1];
  p.vn_sb = v_new->stride[0];
  p.vn_sh = v_new->stride[1];
  p.slots = static_cast<const int64_t*>(slot_mapping->data);
  p.k_cache = static_cast<__nv_bfloat16*>(k_cache->data);
  p.v_cache = static_cast<__nv_bfloat16*>(v_cache->data);
  p.kc_sblk = k_cache->stride[0];
  p.kc_sh = k_cache->stride[1];
  p.vc_sblk = v_cache->stride[0];
  p.vc_sh = v_cache->stride[1];
  p.B = static_cast<int>(B);
  p.Hkv = static_cast<int>(Hkv);
  p.D = static_cast<int>(D);
  p.NB = static_cast<int>(k_cache->shape[0]);
  p.err = err;
  if (forge::launch_append(p, static_cast<cudaStream_t>(stream)) != cudaSuccess) return FORGE_ERR_CUDA;
  return FORGE_OK;
}

int forge_paged_gqa_decode_plan(int B, int Hkv, int max_blocks_per_seq, int split_tokens, int num_sms,
                                int* split_tokens_out, int* kernel_out) {
  if (!split_tokens_out || !kernel_out) return FORGE_ERR_NULL;
  if (B < 0 || Hkv <= 0 || max_blocks_per_seq < 0) return FORGE_ERR_SHAPE;
  if (num_sms <= 0) return FORGE_ERR_VALUE;
  if (split_tokens != 0 &&
      (split_tokens < kMinSplitTokens || split_tokens > kMaxSplitTokens || split_tokens % kBlockSize != 0))
    return FORGE_ERR_VALUE;
  int online = 0;
  const int bps = split_blocks_for(split_tokens, B, Hkv, max_blocks_per_seq, num_sms, &online);
  *split_tokens_out = bps * kBlockSize;
  *kernel_out = online ? FORGE_DECODE_ONLINE : FORGE_DECODE_TWO_PASS;
  return FORGE_OK;
}

size_t forge_paged_gqa_decode_workspace_bytes(int B, int Hq, int Hkv, int D, int max_blocks_per_seq,
                                              int split_tokens) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || max_blocks_per_seq < 0) return 0;
  if (split_tokens != 0 &&
      (split_tokens < kMinSplitTokens || split_tokens > kMaxSplitTokens || split_tokens % kBlockSize != 0))
    return 0;
  // The automatic split length depends on the SM count; plan for the
  // smallest split it can pick so the size is an upper bound.
  const int bps = split_tokens ? split_tokens / kBlockSize : 4;
  const int64_t s_max = max_blocks_per_seq > 0 ? (max_blocks_per_seq + bps - 1) / bps : 1;
  return workspace_bytes_for(B, Hq, D, s_max);
}

int forge_paged_gqa_decode_ex(const forge_tensor* q, const forge_tensor* k_cache, const forge_tensor* v_cache,
                              const forge_tensor* block_tables, const forge_tensor* context_lens, float scale,
                              forge_tensor* out, void* workspace, size_t workspace_bytes, int split_tokens,
                              void* stream) {
  int dev = 0, sms = 0;
  int* err = nullptr;
  DecodePlan plan;
  FORGE_TRY(plan_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out, split_tokens, 148, &plan));
  if (plan.p.B == 0) return FORGE_OK;
  FORGE_TRY(current_device(&dev));
  FORGE_TRY(device_state(dev, &err, &sms));
  if (split_tokens == 0) {  // re-plan with the real SM count
    FORGE_TRY(plan_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out, 0, sms, &plan));
  }
  if (plan.ws_bytes > 0) {
    if (!workspace || workspace_bytes < plan.ws_bytes) return FORGE_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FORGE_ERR_ALIGN;
  }
  plan.p.err = err;
  attach_workspace(&plan, workspace);
  return launch_plan(&plan, static_cast<cudaStream_t>(stream));
}

int forge_paged_gqa_decode(const forge_tensor* q, const forge_tensor* k_cache, const forge_tensor* v_cache,
                           const forge_tensor* block_tables, const forge_tensor* context_lens, float scale,
                           forge_tensor* out, void* stream) {
  DecodePlan plan;
  FORGE_TRY(plan_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out, 0, 148, &plan));
  if (plan.p.B == 0) return FORGE_OK;
  int dev = 0, sms = 0;
  int* err = nullptr;
  FORGE_TRY(current_device(&dev));
  FORGE_TRY(device_state(dev, &err, &sms));
  FORGE_TRY(plan_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out, 0, sms, &plan));
  void* ws = nullptr;
  std::unique_lock<std::mutex> hold;  // the stream's scratch, held until the launch is enqueued
  if (plan.ws_bytes > 0)
    FORGE_TRY(cached_workspace(dev, static_cast<cudaStream_t>(stream), plan.ws_bytes, &ws, &hold));
  plan.p.err = err;
  attach_workspace(&plan, ws);
  return launch_plan(&plan, static_cast<cudaStream_t>(stream));
}

namespace {

// Validates the optional q/k path arguments against head size D.
int check_qk_options(const forge_qk_options* o, int64_t D) {
  if (!o) return FORGE_OK;
  for (const forge_tensor* w : {o->q_norm_weight, o->k_norm_weight}) {
    if (!w) continue;
    FORGE_TRY(check_tensor(w, FORGE_BF16, 1));
    if (w->shape[0] != D) return FORGE_ERR_SHAPE;
    if (!w->data) return FORGE_ERR_NULL;
    if (w->stride[0] != 1) return FORGE_ERR_SHAPE;
  }
  if ((o->q_norm_weight || o->k_norm_weight) && !(std::isfinite(o->norm_eps) && o->norm_eps >= 0.f))
    return FORGE_ERR_VALUE;
  if (o->rope_cos_sin) {
    const forge_tensor* r = o->rope_cos_sin;
    FORGE_TRY(check_tensor(r, FORGE_F32, 2));
    if (r->shape[1] != D || r->shape[0] < 1 || r->shape[0] > INT32_MAX) return FORGE_ERR_SHAPE;
    if (!r->data) return FORGE_ERR_NULL;
    if (r->stride[1] != 1 || r->stride[0] != D) return FORGE_ERR_SHAPE;
  }
  return FORGE_OK;
}

int append_decode_impl(const forge_tensor* q, const forge_tensor* k_new, const forge_tensor* v_new,
                       const forge_qk_options* qk, forge_tensor* k_cache, forge_tensor* v_cache,
                       const forge_tensor* block_tables, const forge_tensor* context_lens, float scale,
                       forge_tensor* out, void* stream);

}  // namespace

int forge_paged_qk_append_gqa_decode(const forge_tensor* q, const forge_tensor* k_new, const forge_tensor* v_new,
                                     const forge_qk_options* qk, forge_tensor* k_cache, forge_tensor* v_cache,
                                     const forge_tensor* block_tables, const forge_tensor* context_lens, float scale,
                                     forge_tensor* out, void* stream) {
  return append_decode_impl(q, k_new, v_new, qk, k_cache, v_cache, block_tables, context_lens, scale, out, stream);
}

int forge_rope_cos_sin_table(double theta, int D, int rows, float* out) {
  if (!out) return FORGE_ERR_NULL;
  if (D <= 0 || D % 2 != 0 || rows <= 0 || !(theta > 0.0)) return FORGE_ERR_VALUE;
  const int h = D / 2;
  for (int i = 0; i < h; ++i) {
    const double inv_freq = std::pow(theta, -2.0 * i / D);
    for (int r = 0; r < rows; ++r) {
      const double a = static_cast<double>(r) * inv_freq;
      out[static_cast<size_t>(r) * D + i] = static_cast<float>(std::cos(a));
      out[static_cast<size_t>(r) * D + h + i] = static_cast<float>(std::sin(a));
    }
  }
  return FORGE_OK;
}

int forge_paged_append_gqa_decode(const forge_tensor* q, const forge_tensor* k_new, const forge_tensor* v_new,
                                  forge_tensor* k_cache, forge_tensor* v_cache, const forge_tensor* block_tables,
                                  const forge_tensor* context_lens, float scale, forge_tensor* out, void* stream) {
  return append_decode_impl(q, k_new, v_new, nullptr, k_cache, v_cache, block_tables, context_lens, scale, out,
                            stream);
}

}  // extern "C"

namespace {

int append_decode_impl(const forge_tensor* q, const forge_tensor* k_new, const forge_tensor* v_new,
                       const forge_qk_options* qk, forge_tensor* k_cache, forge_tensor* v_cache,
                       const forge_tensor* block_tables, const forge_tensor* context_lens, float scale,
                       forge_tensor* out, void* stream) {
  DecodePlan plan;
  FORGE_TRY(plan_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out, 0, 148, &plan));
  FORGE_TRY(check_tensor(k_new, FORGE_BF16, 3));
  FORGE_TRY(check_tensor(v_new, FORGE_BF16, 3));
  for (int i = 0; i < 3; ++i)
    if (v_new->shape[i] != k_new->shape[i]) return FORGE_ERR_SHAPE;
  if (k_new->shape[0] != q->shape[0] || k_new->shape[1] != k_cache->shape[1] || k_new->shape[2] != q->shape[2])
    return FORGE_ERR_SHAPE;
  FORGE_TRY(check_qk_options(qk, q->shape[2]));
  if (plan.p.B == 0) return FORGE_OK;
  FORGE_TRY(check_vec16(k_new, 2));
  FORGE_TRY(check_vec16(v_new, 2));
  int dev = 0, sms = 0;
  int* err = nullptr;
  FORGE_TRY(current_device(&dev));
  FORGE_TRY(device_state(dev, &err, &sms));
  FORGE_TRY(plan_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out, 0, sms, &plan));
  void* ws = nullptr;
  std::unique_lock<std::mutex> hold;  // the stream's scratch, held until the launch is enqueued
  if (plan.ws_bytes > 0)
    FORGE_TRY(cached_workspace(dev, static_cast<cudaStream_t>(stream), plan.ws_bytes, &ws, &hold));
  plan.p.err = err;
  plan.p.k_new = static_cast<const __nv_bfloat16*>(k_new->data);
  plan.p.v_new = static_cast<const __nv_bfloat16*>(v_new->data);
  plan.p.kn_sb = k_new->stride[0];
  plan.p.kn_sh = k_new->stride[1];
  plan.p.vn_sb = v_new->stride[0];
  plan.p.vn_sh = v_new->stride[1];
  plan.p.k_cache_w = static_cast<__nv_bfloat16*>(k_cache->data);
  plan.p.v_cache_w = static_cast<__nv_bfloat16*>(v_cache->data);
  if (qk) {
    if (qk->q_norm_weight) plan.p.q_norm_w = static_cast<const __nv_bfloat16*>(qk->q_norm_weight->data);
    if (qk->k_norm_weight) plan.p.k_norm_w = static_cast<const __nv_bfloat16*>(qk->k_norm_weight->data);
    plan.p.norm_eps = qk->norm_eps;
    if (qk->rope_cos_sin) {
      plan.p.rope = static_cast<const float*>(qk->rope_cos_sin->data);
      plan.p.rope_rows = static_cast<int>(qk->rope_cos_sin->shape[0]);
    }
  }
  attach_workspace(&plan, ws);
  return launch_plan(&plan, static_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

int forge_paged_prefill(const forge_tensor* q, const forge_tensor* k_cache, const forge_tensor* v_cache,
                        const forge_tensor* block_tables, const forge_tensor* context_lens,
                        const forge_tensor* query_start, float scale, forge_tensor* out, void* stream) {
  FORGE_TRY(check_tensor(q, FORGE_BF16, 3));
  FORGE_TRY(check_cache(k_cache));
  FORGE_TRY(check_cache(v_cache));
  FORGE_TRY(check_tensor(block_tables, FORGE_I32, 2));
  FORGE_TRY(check_tensor(context_lens, FORGE_I32, 1));
  FORGE_TRY(check_tensor(query_start, FORGE_I32, 1));
  if (!out) return FORGE_ERR_NULL;
  if (out->dtype != FORGE_BF16 && out->dtype != FORGE_F32) return FORGE_ERR_DTYPE;
  if (out->ndim != 3) return FORGE_ERR_SHAPE;
  const int64_t T = q->shape[0], Hq = q->shape[1], D = q->shape[2];
  const int64_t NB = k_cache->shape[0], Hkv = k_cache->shape[1];
  const int64_t B = context_lens->shape[0], MB = block_tables->shape[1];
  for (int i = 0; i < 4; ++i)
    if (v_cache->shape[i] != k_cache->shape[i]) return FORGE_ERR_SHAPE;
  if (k_cache->shape[3] != D) return FORGE_ERR_SHAPE;
  if (out->shape[0] != T || out->shape[1] != Hq || out->shape[2] != D) return FORGE_ERR_SHAPE;
  if (block_tables->shape[0] != B || query_start->shape[0] != B + 1) return FORGE_ERR_SHAPE;
  if (T > INT32_MAX / 2 || B > INT32_MAX / 2 || Hkv > 65535 || NB > INT32_MAX || MB > (INT32_MAX / kBlockSize))
    return FORGE_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return FORGE_ERR_UNSUPPORTED;
  if (Hkv <= 0 || Hq <= 0) return FORGE_ERR_SHAPE;
  if (Hq % Hkv != 0) return FORGE_ERR_UNSUPPORTED;
  const int64_t G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return FORGE_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return FORGE_ERR_VALUE;
  if (T == 0 || B == 0) return FORGE_OK;
  FORGE_TRY(check_vec16(q, 2));
  FORGE_TRY(check_vec16(out, out->dtype == FORGE_BF16 ? 2 : 4));
  if (!block_tables->data || !context_lens->data || !query_start->data) return FORGE_ERR_NULL;
  if (block_tables->stride[1] != 1 || context_lens->stride[0] != 1 || query_start->stride[0] != 1)
    return FORGE_ERR_SHAPE;
  if (NB > 0 && (!k_cache->data || !v_cache->data)) return FORGE_ERR_NULL;

  int dev = 0, sms = 0;
  int* err = nullptr;
  FORGE_TRY(current_device(&dev));
  FORGE_TRY(device_state(dev, &err, &sms));
  forge::PrefillParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = static_cast<const __nv_bfloat16*>(q->data);
  p.q_st = q->stride[0];
  p.q_sh = q->stride[1];
  p.block_tables = static_cast<const int32_t*>(block_tables->data);
  p.bt_sb = block_tables->stride[0];
  p.context_lens = static_cast<const int32_t*>(context_lens->data);
  p.query_start = static_cast<const int32_t*>(query_start->data);
  p.out = out->data;
  p.o_st = out->stride[0];
  p.o_sh = out->stride[1];
  p.B = static_cast<int>(B);
  p.Hq = static_cast<int>(Hq);
  p.Hkv = static_cast<int>(Hkv);
  p.NB = static_cast<int>(NB);
  p.MB = static_cast<int>(MB);
  p.T = static_cast<int>(T);
  p.qk_scale_log2 = scale * 1.4426950408889634f;
  p.err = err;
  CUtensorMap tmk, tmv;
  FORGE_TRY(encode_cache_map(k_cache, &tmk));
  FORGE_TRY(encode_cache_map(v_cache, &tmv));
  cudaError_t e;
  if (prefill_use_mma_sync()) {
    e = forge::launch_prefill(p, tmk, tmv, static_cast<int>(D), static_cast<int>(G), out->dtype == FORGE_BF16,
                              static_cast<cudaStream_t>(stream));
  } else {
    CUtensorMap tmq;
    FORGE_TRY(encode_q_map(q, static_cast<int>(G), &tmq));
    // Context chunks: an item's attention over more than kPrefillChunkStages
    // stages (4096 tokens) is split into chunks merged in fp32, which bounds
    // the length of each fp32 accumulation (measured on the constructed
    // worst case of the bf16 output's error, all weights rounding the same
    // way and |V| in [7, 8): 0.0158 of the 0.016 bound at 4K tokens in one
    // accumulation, 0.0164 at 16K).  The scratch holds every possible chunk's
    // partial rows; if that would pass kPrefillScratchCap the chunks grow, and
    // without counter slots for every (item, KV head) there is no split.
    void* ws = nullptr;
    std::unique_lock<std::mutex> hold;  // the stream's scratch, held until the launch is enqueued
    const int64_t items = forge::prefill_tc_items(T, B, static_cast<int>(G));
    const int64_t max_stages = (MB * kBlockSize + 127) / 128;
    int64_t C = kPrefillChunkStages;
    auto partial_bytes = [&](int64_t chunks) {
      const int64_t rows = items * Hkv * chunks * forge::kPrefillChunkRows;
      return round256(static_cast<size_t>(rows) * D * 4) + static_cast<size_t>(rows) * 2 * 4;
    };
    while (max_stages > C && kCounterBytes + partial_bytes((max_stages + C - 1) / C) > kPrefillScratchCap) C *= 2;
    if (max_stages > C && items * Hkv <= kCounterSlots) {
      const int64_t chunks = (max_stages + C - 1) / C;
      FORGE_TRY(cached_workspace(dev, static_cast<cudaStream_t>(stream), kCounterBytes + partial_bytes(chunks), &ws,
                                 &hold));
      char* base = static_cast<char*>(ws);
      p.chunk_stages = static_cast<int>(C);
      p.max_chunks = static_cast<int>(chunks);
      p.counters = reinterpret_cast<int*>(base);
      p.ws_o = reinterpret_cast<float*>(base + kCounterBytes);
      p.ws_ml = reinterpret_cast<float*>(base + kCounterBytes +
                                         round256(static_cast<size_t>(items * Hkv * chunks * forge::kPrefillChunkRows) * D * 4));
    }
    e = forge::launch_prefill_tc(p, tmq, tmk, tmv, static_cast<int>(D), static_cast<int>(G),
                                 out->dtype == FORGE_BF16, static_cast<cudaStream_t>(stream));
  }
  return e == cudaSuccess ? FORGE_OK : FORGE_ERR_CUDA;
}

const char* forge_status_string(int status) {
  switch (status) {
    case FORGE_OK: return "FORGE_OK";
    case FORGE_ERR_NULL: return "FORGE_ERR_NULL: a descriptor or needed data pointer is NULL";
    case FORGE_ERR_DTYPE: return "FORGE_ERR_DTYPE: wrong dtype";
    case FORGE_ERR_SHAPE: return "FORGE_ERR_SHAPE: wrong rank, mismatched sizes or unsupported strides";
    case FORGE_ERR_UNSUPPORTED: return "FORGE_ERR_UNSUPPORTED: head size, block size or group size not built";
    case FORGE_ERR_ALIGN: return "FORGE_ERR_ALIGN: pointer or stride breaks 16-byte alignment";
    case FORGE_ERR_CUDA: return "FORGE_ERR_CUDA: a CUDA call or launch failed";
    case FORGE_ERR_WORKSPACE: return "FORGE_ERR_WORKSPACE: workspace missing or too small";
    case FORGE_ERR_VALUE: return "FORGE_ERR_VALUE: scalar argument out of range";
    case FORGE_ERR_CAPACITY: return "FORGE_ERR_CAPACITY: the block pool or the batch has no room";
    default: return "unknown forge status";
  }
}

int forge_paged_get_device_error(void* stream, int* code_out) {
  if (!code_out) return FORGE_ERR_NULL;
  int dev = 0, sms = 0;
  int* err = nullptr;
  FORGE_TRY(current_device(&dev));
  FORGE_TRY(device_state(dev, &err, &sms));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int host = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return FORGE_ERR_CUDA;
  if (cudaMemcpy(&host, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FORGE_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return FORGE_ERR_CUDA;
  *code_out = host;
  return FORGE_OK;
}

const char* forge_paged_version(void) { return "0.1.0"; }

}  // extern "C"
