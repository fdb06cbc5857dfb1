// KV block pool and continuous-batching decode step driver (host), and the
// single-CTA kernel that applies a step to the device block tables.
//
// forge-engine README, "What it implements": the KV cache is a paged block
// allocator with deterministic cleanup, scheduling is continuous, bounded,
// token-budgeted batching, and the sample run ends with zero KV blocks
// allocated.  "Make the Engine Talk", 1.2: every decode pass adds one token
// to each running sequence's cache.  The policies (free stack, FIFO
// admission, preemption of the latest admitted sequence) are spelled out in
// forge_serving.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <deque>
#include <mutex>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "../../include/forge_serving.h"

namespace {

struct SeqBlocks {
  std::vector<int32_t> blocks;  // table row, token order
  int32_t len = 0;
};

int32_t blocks_for(int64_t tokens, int32_t bs) { return static_cast<int32_t>((tokens + bs - 1) / bs); }

}  // namespace

struct forge_kv_pool {
  int32_t num_blocks = 0;
  int32_t block_size = 16;
  int32_t max_blocks_per_seq = 0;
  std::vector<int32_t> free_stack;  // top = back
  std::unordered_map<int64_t, SeqBlocks> seqs;
  mutable std::mutex mu;

  // The *_locked members expect mu to be held.
  int add_locked(int64_t seq_id, int32_t num_tokens) {
    if (num_tokens < 0 || seqs.count(seq_id)) return FORGE_ERR_VALUE;
    const int32_t need = blocks_for(num_tokens, block_size);
    if (need > max_blocks_per_seq) return FORGE_ERR_VALUE;
    if (need > static_cast<int32_t>(free_stack.size())) return FORGE_ERR_CAPACITY;
    SeqBlocks st;
    st.len = num_tokens;
    st.blocks.reserve(static_cast<size_t>(need));
    for (int32_t i = 0; i < need; ++i) {
      st.blocks.push_back(free_stack.back());
      free_stack.pop_back();
    }
    seqs.emplace(seq_id, std::move(st));
    return FORGE_OK;
  }

  // one token at position len; *new_block = the block it opened, or -1
  int grow_locked(int64_t seq_id, int64_t* slot_out, int32_t* new_block) {
    auto it = seqs.find(seq_id);
    if (it == seqs.end()) return FORGE_ERR_VALUE;
    SeqBlocks& st = it->second;
    const int32_t pos = st.len;
    int32_t opened = -1;
    if (pos % block_size == 0) {
      if (static_cast<int32_t>(st.blocks.size()) >= max_blocks_per_seq) return FORGE_ERR_VALUE;
      if (free_stack.empty()) return FORGE_ERR_CAPACITY;
      opened = free_stack.back();
      free_stack.pop_back();
      st.blocks.push_back(opened);
    }
    st.len = pos + 1;
    if (slot_out)
      *slot_out = static_cast<int64_t>(st.blocks[static_cast<size_t>(pos / block_size)]) * block_size +
                  pos % block_size;
    if (new_block) *new_block = opened;
    return FORGE_OK;
  }

  int release_locked(int64_t seq_id) {
    auto it = seqs.find(seq_id);
    if (it == seqs.end()) return FORGE_ERR_VALUE;
    for (auto b = it->second.blocks.rbegin(); b != it->second.blocks.rend(); ++b) free_stack.push_back(*b);
    seqs.erase(it);
    return FORGE_OK;
  }

  int32_t free_locked() const { return static_cast<int32_t>(free_stack.size()); }
};

extern "C" {

forge_kv_pool* forge_kv_pool_create(int32_t num_blocks, int32_t block_size, int32_t max_blocks_per_seq) {
  if (num_blocks < 0 || block_size <= 0 || max_blocks_per_seq <= 0) return nullptr;
  forge_kv_pool* p = new (std::nothrow) forge_kv_pool();
  if (!p) return nullptr;
  try {
    p->num_blocks = num_blocks;
    p->block_size = block_size;
    p->max_blocks_per_seq = max_blocks_per_seq;
    p->free_stack.reserve(static_cast<size_t>(num_blocks));
    for (int32_t i = num_blocks - 1; i >= 0; --i) p->free_stack.push_back(i);  // 0 on top
  } catch (...) {
    delete p;
    return nullptr;
  }
  return p;
}

void forge_kv_pool_destroy(forge_kv_pool* p) { delete p; }

int forge_kv_pool_add(forge_kv_pool* p, int64_t seq_id, int32_t num_tokens) {
  if (!p) return FORGE_ERR_NULL;
  std::lock_guard<std::mutex> lock(p->mu);
  try {
    return p->add_locked(seq_id, num_tokens);
  } catch (...) {
    return FORGE_ERR_CAPACITY;
  }
}

int forge_kv_pool_grow(forge_kv_pool* p, int64_t seq_id, int64_t* slot_out) {
  if (!p) return FORGE_ERR_NULL;
  std::lock_guard<std::mutex> lock(p->mu);
  try {
    return p->grow_locked(seq_id, slot_out, nullptr);
  } catch (...) {
    return FORGE_ERR_CAPACITY;
  }
}

int forge_kv_pool_release(forge_kv_pool* p, int64_t seq_id) {
  if (!p) return FORGE_ERR_NULL;
  std::lock_guard<std::mutex> lock(p->mu);
  return p->release_locked(seq_id);
}

int32_t forge_kv_pool_free_blocks(const forge_kv_pool* p) {
  if (!p) return -1;
  std::lock_guard<std::mutex> lock(p->mu);
  return p->free_locked();
}

int32_t forge_kv_pool_used_blocks(const forge_kv_pool* p) {
  if (!p) return -1;
  std::lock_guard<std::mutex> lock(p->mu);
  return p->num_blocks - p->free_locked();
}

int forge_kv_pool_sequence(const forge_kv_pool* p, int64_t seq_id, int32_t* len_out, int32_t* blocks_out,
                           int32_t capacity, int32_t* nblocks_out) {
  if (!p) return FORGE_ERR_NULL;
  std::lock_guard<std::mutex> lock(p->mu);
  auto it = p->seqs.find(seq_id);
  if (it == p->seqs.end()) return FORGE_ERR_VALUE;
  const SeqBlocks& st = it->second;
  const int32_t n = static_cast<int32_t>(st.blocks.size());
  if (len_out) *len_out = st.len;
  if (nblocks_out) *nblocks_out = n;
  if (blocks_out) {
    if (capacity < n) return FORGE_ERR_SHAPE;
    std::copy(st.blocks.begin(), st.blocks.end(), blocks_out);
  }
  return FORGE_OK;
}

}  // extern "C"

namespace {

struct Request {
  int64_t seq_id;
  int32_t prompt;     // tokens whose K/V the caller writes on admission
  int32_t remaining;  // decode steps still to run
};

struct Event {
  int64_t seq_id;
  int32_t row;
  int32_t tokens;
};

// One pinned host buffer and its device twin; `done` is recorded after the
// apply kernel, which follows the copy that read the host side, so it marks
// both buffers free.
struct Stage {
  int32_t* host = nullptr;
  int32_t* dev = nullptr;
  size_t words = 0;
  cudaEvent_t done = nullptr;
  bool pending = false;
};

constexpr int kStages = 4;

}  // namespace

struct forge_batch {
  forge_kv_pool* pool = nullptr;
  int32_t rows = 0;
  int32_t token_budget = 0;
  std::vector<int64_t> row_seq;      // -1 = empty row
  std::vector<int32_t> row_len;      // context length after the last step (0 = empty)
  std::vector<int64_t> row_slot;     // the last step's slot (-1 = empty)
  std::vector<int32_t> row_new;      // block the last step opened (-1 = none)
  std::vector<int32_t> row_left;     // decode steps still to run
  std::vector<uint64_t> row_order;   // admission counter, for preemption
  std::vector<uint8_t> row_full;     // the device copy of this table row must be rewritten whole
  bool applied = true;               // the last step reached the device
  uint64_t admissions = 0;
  std::deque<Request> waiting;
  std::unordered_set<int64_t> live;  // queued or running
  std::vector<Event> ev[3];          // admitted, retired, preempted (last step)
  std::vector<int32_t> stage;        // the last step, as forge_batch_apply uploads it
  Stage ring[kStages];
  int ring_next = 0;
  int device = -1;
  mutable std::mutex mu;

  void empty_row(int32_t r) {
    row_seq[r] = -1;
    row_len[r] = 0;
    row_slot[r] = -1;
    row_left[r] = 0;
    row_order[r] = 0;
  }

  // Running rows whose next token opens a block.
  int32_t growth_need() const {
    int32_t n = 0;
    for (int32_t r = 0; r < rows; ++r)
      if (row_seq[r] >= 0 && row_len[r] % pool->block_size == 0) ++n;
    return n;
  }

  int step_locked(forge_batch_report* rep);
  void build_stage();
};

// Expects b->mu held; takes the pool's lock itself.
int forge_batch::step_locked(forge_batch_report* rep) {
  std::lock_guard<std::mutex> plock(pool->mu);
  const int32_t bs = pool->block_size;
  for (auto& e : ev) e.clear();
  std::fill(row_new.begin(), row_new.end(), -1);
  if (!applied)  // the previous step never reached the device: resend whole rows
    for (int32_t r = 0; r < rows; ++r)
      if (row_seq[r] >= 0) row_full[r] = 1;

  // 1. retire
  for (int32_t r = 0; r < rows; ++r) {
    if (row_seq[r] >= 0 && row_left[r] == 0) {
      ev[FORGE_BATCH_RETIRED].push_back({row_seq[r], r, row_len[r]});
      pool->release_locked(row_seq[r]);
      live.erase(row_seq[r]);
      empty_row(r);
    }
  }
  // 2. preempt the latest admitted until this step's growth fits
  while (growth_need() > pool->free_locked()) {
    int32_t victim = -1;
    for (int32_t r = 0; r < rows; ++r)
      if (row_seq[r] >= 0 && (victim < 0 || row_order[r] > row_order[victim])) victim = r;
    ev[FORGE_BATCH_PREEMPTED].push_back({row_seq[victim], victim, row_len[victim]});
    pool->release_locked(row_seq[victim]);
    waiting.push_front({row_seq[victim], row_len[victim], row_left[victim]});
    empty_row(victim);
  }
  // 3. admit from the head of the queue
  int64_t admitted_tokens = 0;
  while (!waiting.empty()) {
    const Request& q = waiting.front();
    int32_t row = -1;
    for (int32_t r = 0; r < rows && row < 0; ++r)
      if (row_seq[r] < 0) row = r;
    if (row < 0) break;
    if (!ev[FORGE_BATCH_ADMITTED].empty() && admitted_tokens + q.prompt > token_budget) break;
    if (blocks_for(static_cast<int64_t>(q.prompt) + 1, bs) + growth_need() > pool->free_locked()) break;
    const int rc = pool->add_locked(q.seq_id, q.prompt);
    if (rc != FORGE_OK) return rc;  // cannot happen: checked above
    row_seq[row] = q.seq_id;
    row_len[row] = q.prompt;
    row_left[row] = q.remaining;
    row_order[row] = ++admissions;
    row_full[row] = 1;
    admitted_tokens += q.prompt;
    ev[FORGE_BATCH_ADMITTED].push_back({q.seq_id, row, q.prompt});
    waiting.pop_front();
  }
  // 4. one token for every running row
  int64_t tokens = 0;
  int32_t running = 0;
  for (int32_t r = 0; r < rows; ++r) {
    if (row_seq[r] < 0) continue;
    const int rc = pool->grow_locked(row_seq[r], &row_slot[r], &row_new[r]);
    if (rc != FORGE_OK) return rc;  // cannot happen: the growth was reserved
    row_len[r] += 1;
    row_left[r] -= 1;
    tokens += row_len[r];
    ++running;
  }
  build_stage();
  applied = false;
  if (rep) {
    rep->running = running;
    rep->waiting = static_cast<int32_t>(waiting.size());
    rep->admitted = static_cast<int32_t>(ev[FORGE_BATCH_ADMITTED].size());
    rep->retired = static_cast<int32_t>(ev[FORGE_BATCH_RETIRED].size());
    rep->preempted = static_cast<int32_t>(ev[FORGE_BATCH_PREEMPTED].size());
    rep->free_blocks = pool->free_locked();
    rep->tokens = tokens;
  }
  return FORGE_OK;
}

// Staging layout (int32 words):
//   [0] rows  [1] rows rewritten whole  [2..3] unused
//   [4, 4+rows)          context length per row
//   [4+rows, 4+2*rows)   block opened by this step's token, or -1
//   then per row rewritten whole (admitted by this step, or running while a
//   step went unapplied): row, nblocks, blocks[nblocks]
// Expects both locks held.
void forge_batch::build_stage() {
  stage.clear();
  stage.push_back(rows);
  stage.push_back(0);
  stage.push_back(0);
  stage.push_back(0);
  stage.insert(stage.end(), row_len.begin(), row_len.end());
  stage.insert(stage.end(), row_new.begin(), row_new.end());
  int32_t n_full = 0;
  for (int32_t r = 0; r < rows; ++r) {
    if (!row_full[r] || row_seq[r] < 0) continue;
    const std::vector<int32_t>& blocks = pool->seqs.at(row_seq[r]).blocks;
    stage.push_back(r);
    stage.push_back(static_cast<int32_t>(blocks.size()));
    stage.insert(stage.end(), blocks.begin(), blocks.end());
    ++n_full;
  }
  stage[1] = n_full;
}

namespace {

// One CTA: write the table rows that are resent whole, then (after the
// barrier, so those writes are visible) every row's length, the block its
// new token opened and its slot, read back from the device table.
__global__ void __launch_bounds__(256) batch_apply_kernel(const int32_t* __restrict__ stage, int32_t* tables,
                                                          int64_t table_stride, int32_t table_width,
                                                          int32_t* __restrict__ lens, int64_t* __restrict__ slots,
                                                          int32_t block_size) {
  const int32_t rows = stage[0];
  const int32_t n_full = stage[1];
  const int32_t* len = stage + 4;
  const int32_t* opened = len + rows;
  const int32_t* adm = opened + rows;
  for (int32_t a = 0; a < n_full; ++a) {
    const int32_t row = adm[0];
    const int32_t n = adm[1];
    int32_t* t = tables + row * table_stride;
    for (int32_t c = threadIdx.x; c < table_width; c += blockDim.x) t[c] = c < n ? adm[2 + c] : -1;
    adm += 2 + n;
  }
  __syncthreads();
  for (int32_t r = threadIdx.x; r < rows; r += blockDim.x) {
    const int32_t L = len[r];
    lens[r] = L;
    int64_t slot = -1;
    if (L > 0) {
      int32_t* entry = tables + r * table_stride + (L - 1) / block_size;
      if (opened[r] >= 0) *entry = opened[r];
      slot = static_cast<int64_t>(*entry) * block_size + (L - 1) % block_size;
    }
    slots[r] = slot;
  }
}

void free_stage(Stage& s) {
  if (s.done) {
    cudaEventSynchronize(s.done);
    cudaEventDestroy(s.done);
  }
  if (s.host) cudaFreeHost(s.host);
  if (s.dev) cudaFree(s.dev);
  s = Stage();
}

bool check_vec(const forge_tensor* t, int32_t dtype, int64_t n) {
  return t->ndim == 1 && t->dtype == dtype && t->shape[0] == n && (n <= 1 || t->stride[0] == 1);
}

}  // namespace

extern "C" {

forge_batch* forge_batch_create(forge_kv_pool* pool, int32_t rows, int32_t token_budget) {
  if (!pool || rows <= 0 || token_budget <= 0) return nullptr;
  forge_batch* b = new (std::nothrow) forge_batch();
  if (!b) return nullptr;
  try {
    b->pool = pool;
    b->rows = rows;
    b->token_budget = token_budget;
    b->row_seq.assign(rows, -1);
    b->row_len.assign(rows, 0);
    b->row_slot.assign(rows, -1);
    b->row_new.assign(rows, -1);
    b->row_left.assign(rows, 0);
    b->row_order.assign(rows, 0);
    b->row_full.assign(rows, 0);
    std::lock_guard<std::mutex> plock(pool->mu);
    b->build_stage();
  } catch (...) {
    delete b;
    return nullptr;
  }
  return b;
}

void forge_batch_destroy(forge_batch* b) {
  if (!b) return;
  {
    std::lock_guard<std::mutex> lock(b->mu);
    for (Stage& s : b->ring) free_stage(s);
    std::lock_guard<std::mutex> plock(b->pool->mu);
    for (int32_t r = 0; r < b->rows; ++r)
      if (b->row_seq[r] >= 0) b->pool->release_locked(b->row_seq[r]);
  }
  delete b;
}

int forge_batch_submit(forge_batch* b, int64_t seq_id, int32_t prompt_tokens, int32_t max_new_tokens) {
  if (!b) return FORGE_ERR_NULL;
  std::lock_guard<std::mutex> lock(b->mu);
  const forge_kv_pool* p = b->pool;
  if (prompt_tokens < 0 || max_new_tokens < 1 || b->live.count(seq_id)) return FORGE_ERR_VALUE;
  const int64_t total = static_cast<int64_t>(prompt_tokens) + max_new_tokens;
  const int32_t need = blocks_for(total, p->block_size);
  if (need > p->max_blocks_per_seq) return FORGE_ERR_VALUE;
  if (need > p->num_blocks) return FORGE_ERR_CAPACITY;
  try {
    b->waiting.push_back({seq_id, prompt_tokens, max_new_tokens});
    b->live.insert(seq_id);
  } catch (...) {
    return FORGE_ERR_CAPACITY;
  }
  return FORGE_OK;
}

int forge_batch_step(forge_batch* b, forge_batch_report* report) {
  if (!b) return FORGE_ERR_NULL;
  std::lock_guard<std::mutex> lock(b->mu);
  try {
    return b->step_locked(report);
  } catch (...) {
    return FORGE_ERR_CAPACITY;
  }
}

int forge_batch_rows(const forge_batch* b, int64_t* seq_ids, int32_t* context_lens, int64_t* slots,
                     int32_t* new_blocks) {
  if (!b) return FORGE_ERR_NULL;
  std::lock_guard<std::mutex> lock(b->mu);
  if (seq_ids) std::copy(b->row_seq.begin(), b->row_seq.end(), seq_ids);
  if (context_lens) std::copy(b->row_len.begin(), b->row_len.end(), context_lens);
  if (slots) std::copy(b->row_slot.begin(), b->row_slot.end(), slots);
  if (new_blocks) std::copy(b->row_new.begin(), b->row_new.end(), new_blocks);
  return FORGE_OK;
}

int forge_batch_events(const forge_batch* b, int kind, int32_t capacity, int64_t* seq_ids, int32_t* rows,
                       int32_t* tokens) {
  if (!b) return FORGE_ERR_NULL;
  if (kind < FORGE_BATCH_ADMITTED || kind > FORGE_BATCH_PREEMPTED || capacity < 0) return FORGE_ERR_VALUE;
  std::lock_guard<std::mutex> lock(b->mu);
  const std::vector<Event>& ev = b->ev[kind];
  const size_t n = std::min(ev.size(), static_cast<size_t>(capacity));
  for (size_t i = 0; i < n; ++i) {
    if (seq_ids) seq_ids[i] = ev[i].seq_id;
    if (rows) rows[i] = ev[i].row;
    if (tokens) tokens[i] = ev[i].tokens;
  }
  return static_cast<int>(ev.size());
}

int forge_batch_apply(forge_batch* b, forge_tensor* block_tables, forge_tensor* context_lens,
                      forge_tensor* slot_mapping, void* stream) {
  if (!b || !block_tables || !context_lens || !slot_mapping) return FORGE_ERR_NULL;
  if (!block_tables->data || !context_lens->data || !slot_mapping->data) return FORGE_ERR_NULL;
  std::lock_guard<std::mutex> lock(b->mu);
  const int32_t rows = b->rows;
  if (block_tables->dtype != FORGE_I32 || context_lens->dtype != FORGE_I32 || slot_mapping->dtype != FORGE_I64)
    return FORGE_ERR_DTYPE;
  if (block_tables->ndim != 2 || block_tables->shape[0] != rows ||
      block_tables->shape[1] < b->pool->max_blocks_per_seq || block_tables->stride[1] != 1 ||
      block_tables->stride[0] < block_tables->shape[1] || block_tables->shape[1] > INT32_MAX)
    return FORGE_ERR_SHAPE;
  if (!check_vec(context_lens, FORGE_I32, rows) || !check_vec(slot_mapping, FORGE_I64, rows))
    return FORGE_ERR_SHAPE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return FORGE_ERR_CUDA;
  if (cap != cudaStreamCaptureStatusNone) return FORGE_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FORGE_ERR_CUDA;
  if (b->device < 0) b->device = dev;
  if (b->device != dev) return FORGE_ERR_VALUE;

  Stage& st = b->ring[b->ring_next];
  const size_t words = b->stage.size();
  if (st.pending && cudaEventSynchronize(st.done) != cudaSuccess) return FORGE_ERR_CUDA;
  st.pending = false;
  if (st.words < words) {
    free_stage(st);
    size_t cap_words = 256;
    while (cap_words < words) cap_words *= 2;
    if (cudaHostAlloc(reinterpret_cast<void**>(&st.host), cap_words * sizeof(int32_t), cudaHostAllocDefault) !=
            cudaSuccess ||
        cudaMalloc(reinterpret_cast<void**>(&st.dev), cap_words * sizeof(int32_t)) != cudaSuccess ||
        cudaEventCreateWithFlags(&st.done, cudaEventDisableTiming) != cudaSuccess) {
      free_stage(st);
      return FORGE_ERR_CUDA;
    }
    st.words = cap_words;
  }
  std::copy(b->stage.begin(), b->stage.end(), st.host);
  if (cudaMemcpyAsync(st.dev, st.host, words * sizeof(int32_t), cudaMemcpyHostToDevice, s) != cudaSuccess)
    return FORGE_ERR_CUDA;
  batch_apply_kernel<<<1, 256, 0, s>>>(st.dev, static_cast<int32_t*>(block_tables->data), block_tables->stride[0],
                                       static_cast<int32_t>(block_tables->shape[1]),
                                       static_cast<int32_t*>(context_lens->data),
                                       static_cast<int64_t*>(slot_mapping->data), b->pool->block_size);
  if (cudaGetLastError() != cudaSuccess) return FORGE_ERR_CUDA;
  // One event after the kernel covers both of the stage's buffers: the copy
  // has read the host buffer and the kernel has read the device buffer, so
  // a later apply (on any stream) may refill either.
  if (cudaEventRecord(st.done, s) != cudaSuccess) return FORGE_ERR_CUDA;
  st.pending = true;
  b->ring_next = (b->ring_next + 1) % kStages;
  std::fill(b->row_full.begin(), b->row_full.end(), 0);
  b->applied = true;
  return FORGE_OK;
}

}  // extern "C"
