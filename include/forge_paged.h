/*
 * forge_paged.h -- C ABI of libforge_paged.so: paged-KV append and paged
 * grouped-query-attention decode on NVIDIA GB300 (sm_103a).
 *
 * What the operations are (page title, section):
 *   - forge-engine README, "What it implements", row "KV cache": the KV cache
 *     is a pool of fixed-size blocks handed out by a block allocator; row
 *     "Kernels": decode attention over that cache is a CUDA paged GQA kernel.
 *   - "Make the Engine Talk", 1.2 "The loop behind it": after the prefill,
 *     every decode pass runs the model on ONE new token per sequence and the
 *     cache grows by that token; 1.3 "What the rest of Part I builds": the
 *     attention is grouped-query attention.
 *
 * Definitions (the plain reading where the pages give no formula):
 *   BS = 16 tokens per block.  Token t of sequence b lives in physical block
 *   block_tables[b][t / BS], slot t % BS.  With G = Hq / Hkv, query head h
 *   reads KV head h / G (contiguous groups).  For every b, h:
 *     out[b,h,:] = sum_{t < L_b} softmax_t(scale * q[b,h,:] . K_b[t,:]) V_b[t,:]
 *   with L_b = context_lens[b] (the length AFTER this step's append); out is
 *   zero when L_b == 0.  Cache slots at t >= L_b, free blocks and unused
 *   block-table entries are never read, whatever they hold.
 *
 * Tensors are passed as forge_tensor descriptors (below).  All data pointers
 * are device pointers on the current CUDA device.  The caller owns every
 * tensor; the library keeps no pointer after a call returns.
 *
 * Every call is asynchronous: it validates its arguments on the host,
 * enqueues kernels on `stream` (a cudaStream_t; NULL = the legacy default
 * stream) and returns.  No call reads device memory from the host, so calls
 * can be captured in a CUDA graph (see forge_paged_gqa_decode for its
 * workspace note).  The append and decode kernels are launched with
 * programmatic stream serialization, so their start-up may overlap the end of
 * the previous kernel in the stream.  Before that kernel has completed, a
 * decode kernel only reads its sequence lengths and block-table entries to
 * prefetch its first K/V tiles into L2; it writes nothing and uses no value
 * read then, so stream order holds as for a plain launch.  Calls
 * never abort, throw or trap: they return a forge_status.  Argument errors are reported before anything is enqueued.
 * Violations of the device-side preconditions (a block id outside the pool,
 * a length longer than the table row, a slot outside the pool) make the
 * kernels skip the bad access and record an error code that
 * forge_paged_get_device_error returns.
 */
#ifndef FORGE_PAGED_H
#define FORGE_PAGED_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FORGE_API __attribute__((visibility("default")))
#else
#define FORGE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FORGE_BF16 = 1, /* bfloat16 */
    FORGE_F32 = 2,  /* float32 */
    FORGE_I32 = 3,  /* int32 */
    FORGE_I64 = 4   /* int64 */
} forge_dtype;

/* A strided view of device memory.  shape/stride beyond ndim are ignored.
 * Strides are in ELEMENTS, not bytes. */
typedef struct {
    void *data;
    int32_t dtype; /* forge_dtype */
    int32_t ndim;  /* 1..4 */
    int64_t shape[4];
    int64_t stride[4];
} forge_tensor;

typedef enum {
    FORGE_OK = 0,
    FORGE_ERR_NULL = -1,        /* a descriptor or a needed data pointer is NULL */
    FORGE_ERR_DTYPE = -2,       /* wrong dtype */
    FORGE_ERR_SHAPE = -3,       /* wrong rank, mismatched sizes or unsupported strides */
    FORGE_ERR_UNSUPPORTED = -4, /* valid but not built: D, block size or group size */
    FORGE_ERR_ALIGN = -5,       /* a data pointer or stride breaks 16-byte alignment */
    FORGE_ERR_CUDA = -6,        /* a CUDA runtime call or a launch failed */
    FORGE_ERR_WORKSPACE = -7,   /* workspace NULL or smaller than required */
    FORGE_ERR_VALUE = -8,       /* a scalar argument is out of range (e.g. non-finite scale) */
    FORGE_ERR_CAPACITY = -9     /* a KV block pool or a decode batch has no room (forge_serving.h) */
} forge_status;

/* Device-side error codes (forge_paged_get_device_error). */
#define FORGE_DEVERR_NONE 0
#define FORGE_DEVERR_BLOCK_ID 1   /* a used block-table entry is outside [0, NB) */
#define FORGE_DEVERR_LENGTH 2     /* context_lens[b] > MB * BS (or negative) */
#define FORGE_DEVERR_SLOT 3       /* slot_mapping[b] >= NB * BS */
#define FORGE_DEVERR_TIMEOUT 4    /* a pipeline wait gave up (should never happen) */
#define FORGE_DEVERR_POSITION 5   /* context_lens[b] - 1 beyond the rotary table (rotation skipped) */
#define FORGE_DEVERR_QUERY 6      /* prefill: query_start not 0 at b = 0, decreasing, past T, or n_b > L_b */

/*
 * forge_paged_kv_append -- write this step's new K/V token of every sequence
 * into its cache slot ("Make the Engine Talk", 1.2: each decode pass adds the
 * new token to the cache).
 *
 *   k_new, v_new   bf16 [B, Hkv, D]; innermost stride 1, other strides
 *                  multiples of 8 elements; data 16-byte aligned.
 *   slot_mapping   int64 [B], contiguous.  slot = block * BS + offset.
 *                  A negative slot skips that row (padding).  Two rows with
 *                  the same non-negative slot are a precondition violation
 *                  (which row wins is undefined).  slot >= NB*BS is skipped
 *                  and flagged FORGE_DEVERR_SLOT.
 *   k_cache,
 *   v_cache        bf16 [NB, Hkv, BS, D], modified in place.  BS must be 16.
 *                  stride[3] == 1 and stride[2] == D (each (block, head)
 *                  tile is one contiguous BS*D run); stride[0], stride[1]
 *                  multiples of 8 elements; data 16-byte aligned.
 *   stream         cudaStream_t to enqueue on.
 *
 * Supported: D a multiple of 8 (any D the decode supports).  The copy is
 * bit-exact.  Nothing but the addressed slots changes.
 */
FORGE_API int forge_paged_kv_append(const forge_tensor *k_new, const forge_tensor *v_new,
                          const forge_tensor *slot_mapping, forge_tensor *k_cache,
                          forge_tensor *v_cache, void *stream);

/*
 * forge_paged_gqa_decode -- grouped-query attention of one query token per
 * sequence over that sequence's paged K/V (forge-engine README, "What it
 * implements", row "Kernels": CUDA paged GQA; definition at the top of this
 * file).
 *
 *   q              bf16 [B, Hq, D]; innermost stride 1; data 16-B aligned;
 *                  strides multiples of 8 elements.
 *   k_cache,
 *   v_cache        bf16 [NB, Hkv, BS, D] with the layout rules of append.
 *   block_tables   int32 [B, MB]; stride[1] == 1.  Entries past a
 *                  sequence's last block are never read (any value).
 *   context_lens   int32 [B], contiguous.  0 <= L_b <= MB * BS.
 *   scale          logit scale (finite), e.g. 1/sqrt(D).
 *   out            [B, Hq, D] bf16 (rounded to nearest even) or f32;
 *                  innermost stride 1; strides multiples of 8 elements.
 *   stream         cudaStream_t.
 *
 * Supported: D in {64, 128}; BS = 16; G = Hq/Hkv in {1, 2, 4, 8}.
 * Work is split along the context in splits of up to 1024 tokens (shorter
 * when B * Hkv is small against the SM count); for a sequence with more than
 * one split, the last split to finish merges them.  Two kernels compute the
 * same result: a two-pass one per split (logits staged in shared memory) and
 * a single-pass online-softmax one; forge_paged_gqa_decode_plan states which
 * one a call uses and how long its splits are.  Every decode entry point of
 * this header uses the same choice.
 * Arithmetic: products of bf16 values on the tensor cores with fp32
 * accumulation; softmax, sums and the split merge in fp32.  The softmax
 * weights enter the P V product as bf16 high + low parts (about 16
 * significant bits) whatever the output type, so the error of the result
 * before its final rounding stays near 1e-5 of max|V|.  The parity tests
 * hold the result within 2e-3 (f32 out) or 1.6e-2 (bf16 out) max-abs of
 * exact attention, including a case built to make rounded weights fail
 * (outputs near 7.5, where bf16's own rounding is up to 2^-6).
 * Split scratch: a per-(device, stream) buffer that the library owns.  It is
 * allocated on first need and grown when a larger problem arrives, in stream
 * order on `stream` (cudaMallocAsync, zero-filled by cudaMemsetAsync; the old
 * buffer goes back with cudaFreeAsync after the work queued before it), so no
 * call synchronises the host.  While `stream` is being captured into a CUDA
 * graph the scratch cannot grow: such a call returns FORGE_ERR_WORKSPACE
 * before enqueuing anything, so make the first call of the largest size on a
 * stream before capturing it.  Use forge_paged_gqa_decode_ex to pass
 * caller-owned scratch instead.  Thread-safe, also for several host threads
 * on one stream: a call holds its stream's scratch from lookup until its
 * kernel is enqueued.
 */
FORGE_API int forge_paged_gqa_decode(const forge_tensor *q, const forge_tensor *k_cache,
                           const forge_tensor *v_cache, const forge_tensor *block_tables,
                           const forge_tensor *context_lens, float scale, forge_tensor *out,
                           void *stream);

/*
 * Bytes of split scratch that forge_paged_gqa_decode_ex needs for these
 * sizes and split length (split_tokens a multiple of 16 in [16, 1024]).
 * split_tokens = 0 returns an upper bound valid for the automatic split
 * length.  Returns 0 when no scratch is needed (one split per sequence) or
 * the sizes are invalid.  Host-only, no CUDA call.
 */
FORGE_API size_t forge_paged_gqa_decode_workspace_bytes(int B, int Hq, int Hkv, int D,
                                              int max_blocks_per_seq, int split_tokens);

/* Decode kernels a plan can choose (forge_paged_gqa_decode_plan). */
#define FORGE_DECODE_TWO_PASS 0 /* logits of a split staged in shared memory, then P V */
#define FORGE_DECODE_ONLINE 1   /* single pass, running max and sum per head */

/*
 * The split length and kernel that the decode entry points use for these
 * sizes on a GPU with num_sms SMs (num_sms > 0).  split_tokens as for
 * forge_paged_gqa_decode_ex (0 = automatic).  Automatic length: the longest
 * split from 1024 tokens, halving down to 64, whose upper bound on CTAs
 * (B * Hkv * ceil(max_blocks_per_seq * 16 / split)) reaches 4 * num_sms.
 * Kernel: FORGE_DECODE_ONLINE; the environment variable FORGE_DECODE_KERNEL
 * ("online" / "two_pass") overrides it (an automatic two-pass split is at
 * most 512 tokens).  Writes *split_tokens_out and *kernel_out; returns
 * FORGE_OK, FORGE_ERR_NULL, FORGE_ERR_VALUE (bad split_tokens or num_sms) or
 * FORGE_ERR_SHAPE (negative sizes).  Host-only, no CUDA call.
 */
FORGE_API int forge_paged_gqa_decode_plan(int B, int Hkv, int max_blocks_per_seq, int split_tokens,
                                          int num_sms, int *split_tokens_out, int *kernel_out);

/*
 * forge_paged_gqa_decode_ex -- forge_paged_gqa_decode with caller-owned
 * scratch (device memory, 256-byte aligned, at least
 * forge_paged_gqa_decode_workspace_bytes(...) bytes; may be NULL only when
 * that size is 0) and an explicit split length in tokens (0 = automatic,
 * else a multiple of 16 in [16, 1024]).  Allocates nothing.  The first 256
 * KiB of a workspace hold split arrival counters (one per sequence and KV
 * head, so B * Hkv <= 65536 whenever scratch is needed): zero-fill the
 * workspace once before its first use; every completed call leaves the
 * counters at zero and writes nothing else there, so one workspace may then
 * serve calls of any shape without clearing.  Calls that share one workspace
 * must not overlap on the GPU.
 */
FORGE_API int forge_paged_gqa_decode_ex(const forge_tensor *q, const forge_tensor *k_cache,
                              const forge_tensor *v_cache, const forge_tensor *block_tables,
                              const forge_tensor *context_lens, float scale, forge_tensor *out,
                              void *workspace, size_t workspace_bytes, int split_tokens,
                              void *stream);

/*
 * forge_paged_append_gqa_decode -- this step's append and decode in one
 * launch.  Same result as forge_paged_kv_append with each sequence's new
 * token at position context_lens[b] - 1 (slot taken from its block table:
 * block_tables[b][(L_b-1)/BS] * BS + (L_b-1) % BS) followed by
 * forge_paged_gqa_decode ("Make the Engine Talk", 1.2: each decode pass
 * adds the one new token to the cache and attends over everything cached).
 *
 *   q, k_cache, v_cache, block_tables, context_lens, scale, out, stream:
 *                  as forge_paged_gqa_decode (caches are written).
 *   k_new, v_new   bf16 [B, Hkv, D], layout rules of forge_paged_kv_append.
 *
 * A sequence with L_b = 0 appends nothing.  The kernel that reads the
 * sequence's last block writes the new row into it (in shared memory and in
 * the cache), so no other launch is needed; the block holding position
 * L_b - 1 must not be read by another sequence of the same call.  Scratch,
 * its growth and thread-safety as in forge_paged_gqa_decode (library-owned).
 */
FORGE_API int forge_paged_append_gqa_decode(const forge_tensor *q, const forge_tensor *k_new,
                                  const forge_tensor *v_new, forge_tensor *k_cache,
                                  forge_tensor *v_cache, const forge_tensor *block_tables,
                                  const forge_tensor *context_lens, float scale, forge_tensor *out,
                                  void *stream);

/*
 * The q/k path before attention ("Make the Engine Talk", 1.3: RMSNorm and
 * rotary position embeddings are mechanisms of the forward pass), applied to
 * each query head row and to each new key row of the fused call below, at the
 * new token's position pos = context_lens[b] - 1:
 *   x <- x / sqrt(mean(x^2) + norm_eps) * weight          (when a weight is set)
 *   for i < D/2, with (c, s) = rope_cos_sin[pos][i], [pos][D/2 + i]:
 *     x[i] <- x[i] c - x[i + D/2] s,  x[i + D/2] <- x[i + D/2] c + x[i] s
 * computed in fp32 and rounded once to bf16.  The rotated key is what the
 * cache stores.
 *
 *   q_norm_weight,
 *   k_norm_weight  bf16 [D], contiguous, or NULL (no RMSNorm on that side).
 *   norm_eps       >= 0, finite (used when a weight is set).
 *   rope_cos_sin   f32 [P, D], contiguous: cos of pos * theta^(-2i/D) in
 *                  columns [0, D/2), sin in [D/2, D); see
 *                  forge_rope_cos_sin_table.  NULL: no rotation.  A position
 *                  >= P skips the rotation and records FORGE_DEVERR_POSITION.
 */
typedef struct {
    const forge_tensor *q_norm_weight;
    const forge_tensor *k_norm_weight;
    float norm_eps;
    const forge_tensor *rope_cos_sin;
} forge_qk_options;

/*
 * forge_paged_qk_append_gqa_decode -- forge_paged_append_gqa_decode with the
 * q/k path above applied to q and k_new inside the same launch (qk may be
 * NULL: then identical to forge_paged_append_gqa_decode).
 */
FORGE_API int forge_paged_qk_append_gqa_decode(const forge_tensor *q, const forge_tensor *k_new,
                                     const forge_tensor *v_new, const forge_qk_options *qk,
                                     forge_tensor *k_cache, forge_tensor *v_cache,
                                     const forge_tensor *block_tables,
                                     const forge_tensor *context_lens, float scale,
                                     forge_tensor *out, void *stream);

/*
 * Fill out[rows * D] (host memory, f32) with the rotary table for
 * forge_qk_options.rope_cos_sin: out[r][i] = cos(r * theta^(-2i/D)) and
 * out[r][D/2 + i] = sin(r * theta^(-2i/D)) for i < D/2, computed in double.
 * Host-only, no CUDA call.  FORGE_ERR_VALUE for D odd or <= 0, rows <= 0 or
 * theta <= 0.
 */
FORGE_API int forge_rope_cos_sin_table(double theta, int D, int rows, float *out);

/*
 * forge_paged_gqa_decode_noalloc -- forge_paged_gqa_decode for callers that
 * must not allocate device memory.  (The pages have no counterpart: this is
 * an entry point of this library only.)
 *
 * Who needs it: processes that fix their device memory at start-up and
 * must not allocate later -- a serving loop that handed everything left over
 * to its KV-block pool, where a later allocation fails or evicts cache
 * blocks -- and callers that run under a memory manager of their own (an
 * embedding runtime or framework allocator) that forbids allocations it did
 * not make.  forge_paged_gqa_decode may allocate its split scratch on first
 * use; this call never calls cudaMalloc, cudaMallocAsync, cudaFree or any
 * other allocating routine.
 *
 * Arguments, layouts, results and errors are those of forge_paged_gqa_decode.
 * The split scratch is a static device array of FORGE_NOALLOC_SCRATCH_BYTES
 * (16 MiB) inside the library, which every GPU that loads the library holds
 * until the process exits.  The call uses the automatic split length if its
 * scratch fits there, else 1024-token splits; if even those need more, it
 * returns FORGE_ERR_WORKSPACE before enqueuing anything.  (At 32 query
 * heads and D 128, 16 MiB covers batch 32 with block tables of up to 16K
 * tokens; it needs about B * Hq * ceil(table tokens / split) * (D + 2) * 4
 * bytes.)
 *
 * The first call on a device looks up the array's device address (a
 * cudaGetSymbolAddress, with that device current) and caches it; make that
 * first call before any stream capture.  Every call on a device shares the one
 * array and leaves its contents behind.  The only part that must start at
 * zero, the split arrival counters, is zero when the library loads (static
 * device memory) and every completed call returns it to zero; all other
 * scratch values are written before they are read.  Calls that overlap on the
 * GPU (other streams, other threads) race on the array: serialise them.
 */
#define FORGE_NOALLOC_SCRATCH_BYTES (16u << 20)
FORGE_API int forge_paged_gqa_decode_noalloc(const forge_tensor *q, const forge_tensor *k_cache,
                                   const forge_tensor *v_cache, const forge_tensor *block_tables,
                                   const forge_tensor *context_lens, float scale, forge_tensor *out,
                                   void *stream);

/*
 * forge_paged_prefill -- causal attention of a run of new query tokens per
 * sequence over its paged cache ("Make the Engine Talk", 1.2: the prefill
 * runs one forward pass over all of a prompt's tokens at once and fills the
 * cache; chunked, the run is the next piece of a longer context).  The run's
 * K/V must already be in the cache (forge_paged_kv_append with one slot per
 * token).  For sequence b with n_b = query_start[b+1] - query_start[b] query
 * tokens and L_b = context_lens[b] cached tokens (the run included), query
 * row query_start[b] + i sits at position p = L_b - n_b + i and
 *   out[row, h, :] = sum_{t <= p} softmax_t(scale * q[row, h, :] . K_b[t, h/G, :]) V_b[t, h/G, :]
 * with K_b / V_b addressed through block_tables as in the decode (which is
 * the n_b = 1 case).
 *
 *   q             bf16 [T, Hq, D]; last dim contiguous, 16-byte aligned, other
 *                 strides multiples of 8 elements.
 *   k_cache,
 *   v_cache       bf16 [NB, Hkv, 16, D] (as for the decode).
 *   block_tables  int32 [B, MB], inner stride 1.
 *   context_lens  int32 [B], contiguous: L_b, at most MB * 16.
 *   query_start   int32 [B + 1], contiguous: 0 = query_start[0] <= ... <=
 *                 query_start[B] <= T; 0 <= n_b <= L_b.
 *   scale         finite.
 *   out           f32 or bf16 [T, Hq, D], strides as q; rows outside every
 *                 sequence's range are left as they are.
 * D in {64, 128}, Hq / Hkv in {1, 2, 4, 8}.  Enqueues one kernel on `stream`
 * and returns without syncing.  A query_start or length that breaks the rules
 * above is recorded as FORGE_DEVERR_QUERY / FORGE_DEVERR_LENGTH and that
 * sequence's rows are not written; a bad block id as FORGE_DEVERR_BLOCK_ID.
 *
 * Long contexts: when block_tables can address more than 4096 tokens
 * (MB * 16 > 4096), each piece of work whose context passes 4096 tokens is
 * split into context chunks of at most 4096 tokens that run in parallel and
 * are merged in fp32, so that no single fp32 accumulation runs over more than
 * 4096 tokens (over 8K and more tokens the bf16 output can pass the 1.6e-2
 * bound in the worst case).  The chunks' partial rows live in the same
 * library-owned, stream-ordered scratch as the decode's split partials (see
 * forge_paged_gqa_decode: grown on demand with cudaMallocAsync on `stream`,
 * FORGE_ERR_WORKSPACE if it must grow while `stream` is being captured;
 * make one call of the largest shape first).  It is sized for every possible
 * chunk, T / (256 / G) + B pieces x Hkv x ceil(MB * 16 / 4096) chunks x 256
 * rows x (D + 2) x 4 bytes, and is capped at 1 GiB by lengthening the chunks.
 * With block tables of at most 4096 tokens no scratch is used and the call
 * allocates nothing.  (The FORGE_PREFILL_KERNEL=mma kernel does not split.)
 */
FORGE_API int forge_paged_prefill(const forge_tensor *q, const forge_tensor *k_cache,
                                  const forge_tensor *v_cache, const forge_tensor *block_tables,
                                  const forge_tensor *context_lens, const forge_tensor *query_start,
                                  float scale, forge_tensor *out, void *stream);

/* Human-readable name of a forge_status.  Never NULL. */
FORGE_API const char *forge_status_string(int status);

/*
 * Read and clear the device-side error code (FORGE_DEVERR_*) of the current
 * device.  Synchronises `stream` first, so it reports errors of work enqueued
 * before it.  Returns FORGE_OK or FORGE_ERR_CUDA / FORGE_ERR_NULL.
 */
FORGE_API int forge_paged_get_device_error(void *stream, int *code_out);

/* Library version, e.g. "0.1.0". */
FORGE_API const char *forge_paged_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FORGE_PAGED_H */
