// kvq_host.cu — the C ABI of libkvq (include/kvq.h): argument validation,
// handle lifetime, the rotation bank, launches, the device status word and the
// kernel-timing record.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <new>

#include "kvq_internal.cuh"

struct kvq_handle {
  kvq_layout L;
  int G = 4;
  float sm_scale = 0.f;
  int device = 0;
  int num_sms = 1;
  int ctas_int2 = 1, ctas_bf16 = 1;
  int ctas_prep[4] = {1, 1, 1, 1};  // step-preparation CTAs per SM, 1/2/4/8 sequences each
  uint32_t* status = nullptr;      // device
  float* bank = nullptr;           // device: R [2][Hkv][D][D], RVt [Hkv][D][D], mu [Hkv][D]
  bool ready = false;
  // kernel timing
  bool prof = false;
  static constexpr int kSlots = 256;
  cudaEvent_t ev[kSlots][2] = {};
  bool pending[kSlots] = {};
  int next = 0;
  double total_ms = 0.0;
  int launches = 0;
};

namespace {

using kvq::kDim;
using kvq::kPage;

bool layout_ok(const kvq_layout* L) {
  if (!L) return false;
  if (L->head_dim != kDim || L->group != kDim || L->page_size != kPage) return false;
  if (L->num_kv_heads < 1 || L->num_kv_heads > 64) return false;
  if (L->num_heads < 1 || L->num_heads % L->num_kv_heads != 0) return false;
  const int G = L->num_heads / L->num_kv_heads;
  if (G != 1 && G != 2 && G != 4) return false;
  if (!(L->clip_k > 0.f && L->clip_k <= 1.f) || !(L->clip_v > 0.f && L->clip_v <= 1.f))
    return false;
  if (!(L->sm_scale == L->sm_scale)) return false;        // NaN
  if (L->flags & ~(KVQ_OUT_ROTATED | KVQ_Q_ROTATED)) return false;
  return true;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? KVQ_OK : KVQ_ECUDA; }

cudaStream_t S(void* s) { return reinterpret_cast<cudaStream_t>(s); }

size_t rot_floats(int Hkv) {
  return static_cast<size_t>(3) * Hkv * kDim * kDim + static_cast<size_t>(Hkv) * kDim;
}

// KV heads served by one INT2 decode CTA: the largest of 8, 4, 2, 1 dividing Hkv.
int heads_per_cta(int Hkv) {
  for (int c = kvq::kInt2Warps; c > 1; c >>= 1)
    if (Hkv % c == 0) return c;
  return 1;
}

// Heads per CTA for a decode with a given split count: the largest divisor of
// Hkv (at most 8) whose grid fills the GPU's CTA slots best, so that a small
// batch with a fixed split count (one 128K sequence over 64 splits: 64 CTAs of
// 8 heads on 152 SMs) spreads its heads over more CTAs.  Fewer heads per CTA
// means more warps per head and a shared-memory merge of their partials; a
// count is only taken if each warp still gets at least 16 pages (four stages)
// of a full chunk.
int heads_per_cta_for(const kvq_handle* h, int batch, int splits, int chunk_pages) {
  const int Hkv = h->L.num_kv_heads;
  const long slots = static_cast<long>(h->num_sms) * h->ctas_int2;
  const int c_max = heads_per_cta(Hkv);
  int best = c_max;
  double best_fill = -1.0;
  for (int c = c_max; c >= 1; c >>= 1) {
    if (Hkv % c) continue;
    if (c != c_max && chunk_pages * c < 16 * kvq::kInt2Warps) continue;
    const long ctas = static_cast<long>(splits) * (Hkv / c) * batch;
    const long waves = (ctas + slots - 1) / slots;
    const double fill = static_cast<double>(ctas) / static_cast<double>(waves * slots);
    if (fill > best_fill + 0.05) {       // a smaller c must fill clearly better
      best_fill = fill;
      best = c;
    }
  }
  return best;
}

long decode_units(const kvq_handle* h, int batch, bool int2) {
  const int Hkv = h->L.num_kv_heads;
  return static_cast<long>(batch) * (int2 ? Hkv / heads_per_cta(Hkv) : Hkv);
}

// Upper bound of the automatic split count for `batch` sequences (sizes the
// workspace): up to four waves of CTAs.
int splits_cap(const kvq_handle* h, int batch, bool int2) {
  const long units = decode_units(h, batch, int2);
  const long slots = static_cast<long>(h->num_sms) * (int2 ? h->ctas_int2 : h->ctas_bf16);
  long s = (4 * slots) / units;
  if (s < 1) s = 1;
  if (s > kvq::kMaxSplits) s = kvq::kMaxSplits;
  return static_cast<int>(s);
}

// Automatic split count: the number of full waves (1..4) of CTAs that fills the
// GPU best, never with fewer than 8 pages per split.
int choose_splits(const kvq_handle* h, int batch, int max_pages, bool int2,
                  bool window = false) {
  const long units = decode_units(h, batch, int2);
  const long slots = static_cast<long>(h->num_sms) * (int2 ? h->ctas_int2 : h->ctas_bf16);
  const int by_pages = (max_pages + 7) / 8;
  int best = 1;
  double best_fill = -1.0;
  for (int waves = 1; waves <= 4; ++waves) {
    long s = (waves * slots) / units;
    if (s < 1) s = 1;
    if (s > by_pages) s = by_pages;
    if (s > kvq::kMaxSplits) s = kvq::kMaxSplits;
    const long ctas = s * units;
    const long used_waves = (ctas + slots - 1) / slots;
    const double fill = static_cast<double>(ctas) / static_cast<double>(used_waves * slots);
    if (fill > best_fill + 1e-9) {
      best_fill = fill;
      best = static_cast<int>(s);
    }
  }
  if (best < 1) best = 1;
  // Several sequences whose chunks take more than one wave get the balanced
  // schedule (decode_common), whose chunks fill whole waves by construction:
  // two waves (measured on the 64-sequence ragged batch: 173.5 us per step
  // against 176.0 with one wave and 184.5 with four).
  if (int2 && !window && batch >= 2 && units * best > slots) {
    long s = (2 * slots + units - 1) / units;
    if (s > kvq::kMaxSplits) s = kvq::kMaxSplits;
    best = static_cast<int>(s < 1 ? 1 : s);
  }
  return best;
}

void prof_begin(kvq_handle* h, cudaStream_t st, int* slot) {
  *slot = -1;
  if (!h->prof) return;
  const int k = h->next;
  h->next = (h->next + 1) % kvq_handle::kSlots;
  if (h->pending[k]) {          // fold the slot's previous (long finished) pair in
    float ms = 0.f;
    cudaEventSynchronize(h->ev[k][1]);
    if (cudaEventElapsedTime(&ms, h->ev[k][0], h->ev[k][1]) == cudaSuccess) h->total_ms += ms;
    h->pending[k] = false;
  }
  if (!h->ev[k][0]) {
    if (cudaEventCreate(&h->ev[k][0]) != cudaSuccess || cudaEventCreate(&h->ev[k][1]) != cudaSuccess)
      return;
  }
  cudaEventRecord(h->ev[k][0], st);
  *slot = k;
}

void prof_end(kvq_handle* h, cudaStream_t st, int slot) {
  if (slot < 0) return;
  cudaEventRecord(h->ev[slot][1], st);
  h->pending[slot] = true;
  h->launches += 1;
}

int check_decode_args(kvq_handle* h, const void* pool, int num_pool_pages, const uint16_t* q,
                      const int32_t* page_table, int max_pages, const int32_t* seq_lens,
                      int batch, float* out, void* workspace, int num_splits) {
  if (!h || !pool || !q || !page_table || !seq_lens || !out || !workspace) return KVQ_EINVAL;
  if (num_pool_pages < 1 || max_pages < 1 || batch < 1 || batch > 65535) return KVQ_EINVAL;
  if (num_splits < 0 || num_splits > kvq::kMaxSplits) return KVQ_EINVAL;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return KVQ_EINVAL;
  if (reinterpret_cast<uintptr_t>(pool) % 16 != 0) return KVQ_EINVAL;
  if (reinterpret_cast<uintptr_t>(q) % 4 != 0) return KVQ_EINVAL;
  return KVQ_OK;
}

// The BF16 window of kvq_decode_window (absent for the plain decodes).
struct Window {
  const void* bf16_pool = nullptr;
  int bf16_num_pool_pages = 0;
  const int32_t* bf16_page_table = nullptr;
  int sink = 0, recent = 0;
  bool on = false;
};

int decode_common(kvq_handle* h, bool int2, const void* pool, int num_pool_pages,
                  const uint16_t* q, const int32_t* page_table, int max_pages,
                  const int32_t* seq_lens, int batch, float* out, void* workspace,
                  size_t ws_bytes, int num_splits, void* stream, const Window& win = Window(),
                  kvq::StepArgs* step = nullptr) {
  int rc = check_decode_args(h, pool, num_pool_pages, q, page_table, max_pages, seq_lens, batch,
                             out, workspace, num_splits);
  if (rc != KVQ_OK) return rc;
  if (win.on) {
    if (h->L.flags & KVQ_Q_ROTATED) return KVQ_EINVAL;
    if (!win.bf16_pool || !win.bf16_page_table || win.bf16_num_pool_pages < 1) return KVQ_EINVAL;
    if (win.sink < 0 || win.recent < 0) return KVQ_EINVAL;
    if (reinterpret_cast<uintptr_t>(win.bf16_pool) % 16 != 0) return KVQ_EINVAL;
  }
  if (int2 && !h->ready) return KVQ_ENOTREADY;
  const int splits = num_splits ? num_splits : choose_splits(h, batch, max_pages, int2, win.on);
  const kvq::DecodeWs w =
      kvq::decode_ws_layout(batch, h->L.num_kv_heads, h->L.num_heads, splits, int2);
  if (ws_bytes < w.total) return KVQ_ENOSPACE;
  kvq::DeviceGuard dev_guard(h->device);
  if (!dev_guard.ok()) return KVQ_ECUDA;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  kvq::DecodeArgs a;
  a.pool = static_cast<const uint8_t*>(pool);
  a.num_pool_pages = num_pool_pages;
  a.q = q;
  a.page_table = page_table;
  a.max_pages = max_pages;
  a.seq_lens = seq_lens;
  a.batch = batch;
  a.H = h->L.num_heads;
  a.Hkv = h->L.num_kv_heads;
  a.G = h->G;
  a.splits = splits;
  a.chunk_pages = (max_pages + splits - 1) / splits;
  a.qfrag = reinterpret_cast<const uint32_t*>(ws + w.qfrag_off);
  a.qmeta = reinterpret_cast<const float*>(ws + w.qmeta_off);
  a.part = reinterpret_cast<float*>(ws + w.part_off);
  // a balanced schedule (below) keeps the most KV heads per CTA: its chunks fill
  // whole waves whatever the head grouping
  const bool multi_wave = int2 && !win.on && batch >= 2 &&
                          static_cast<long>(batch) * splits * (a.Hkv / heads_per_cta(a.Hkv)) >
                              static_cast<long>(h->num_sms) * h->ctas_int2;
  a.hpc = int2 ? (multi_wave ? heads_per_cta(a.Hkv) : heads_per_cta_for(h, batch, splits, a.chunk_pages))
               : heads_per_cta(a.Hkv);
  a.out = out;
  a.RVt = h->bank ? h->bank + static_cast<size_t>(2) * a.Hkv * kDim * kDim : nullptr;
  a.RV = h->bank ? h->bank + static_cast<size_t>(a.Hkv) * kDim * kDim : nullptr;
  a.rotate_out = (int2 && !(h->L.flags & KVQ_OUT_ROTATED)) ? 1 : 0;
  // one combine CTA per query head when those CTAs fit in one wave (measured:
  // 36-layer stack at 8K 23.7 -> 22.8 us per layer, one 128K sequence over 256
  // splits 49.5 -> 38.9 us per step)
  // Length-balanced chunks when several sequences' chunks take more than one
  // wave of decode CTAs: the batch * splits CTAs are then shared out in
  // proportion to the sequences' lengths (equal lengths give the plain chunks;
  // measured on the 64-sequence ragged batch: decode kernel 188 -> 152 us).
  if (int2) {
    a.sched_map = reinterpret_cast<int4*>(ws + w.sched_off);
    a.sched_nsplit = reinterpret_cast<int*>(ws + w.sched_off + static_cast<size_t>(batch) * splits * 16);
    a.sched_base = a.sched_nsplit + batch;
    const long slots = static_cast<long>(h->num_sms) * h->ctas_int2;
    const long ctas = static_cast<long>(batch) * splits * (a.Hkv / a.hpc);
    a.balanced = multi_wave ? 1 : 0;
    // whole waves only: chunks of one size that spill a few CTAs into a last,
    // partial wave would double the makespan
    a.sched_ctas = a.balanced ? static_cast<int>((ctas / slots) * slots / (a.Hkv / a.hpc)) : 0;
  }
  // Sequences per append CTA of the step preparation: the fewest (1, 2, 4 or
  // 8) that bring its ceil(batch / nb) * Hkv * (2 + nb / min(nb, 2)) CTAs (key
  // append, value append, queries two sequences at a time; each stages one
  // rotation matrix) down to one wave, so that a large batch neither stages
  // the rotations once per sequence nor runs its preparation in several waves.
  a.prep_nb = 1;
  for (int k = 0; k < 3; ++k) {
    const long roles = 2 + (a.prep_nb < 2 ? 1 : a.prep_nb / 2);
    const long ctas = roles * ((batch + a.prep_nb - 1) / a.prep_nb) * a.Hkv;
    if (ctas <= static_cast<long>(h->num_sms) * h->ctas_prep[k]) break;
    a.prep_nb *= 2;
  }
  // the KV-head combine in small CTAs (four per SM, R_V^T read from L2) when
  // one 512-thread CTA per SM would take more than a wave (64-sequence ragged
  // step: 165.3 -> 163.1 us; at batch 16 x 8 KV heads, one wave either way,
  // the 512-thread CTAs with R_V^T staged are faster: 82.8 vs 84.1 us)
  a.combine_small = (!win.on &&
                     static_cast<long>(batch) * a.Hkv > h->num_sms) ? 1 : 0;
  a.combine_per_head =
      (int2 && !win.on &&
       static_cast<long>(batch) * a.Hkv * a.G <=
           static_cast<long>(h->num_sms) * kvq::combine_head_ctas_per_sm())
          ? 1
          : 0;
  a.status = h->status;
  a.log2_scale = h->sm_scale * 1.4426950408889634f;
  a.window = win.on ? 1 : 0;
  a.win_sink = win.on ? win.sink : 0;
  a.win_recent = win.on ? win.recent : 0;
  a.bf16_pool = static_cast<const uint8_t*>(win.bf16_pool);
  a.bf16_num_pool_pages = win.bf16_num_pool_pages;
  a.bf16_page_table = win.bf16_page_table;
  cudaStream_t st = S(stream);
  cudaError_t e;
  if (int2) {
    const float* mu = h->bank + static_cast<size_t>(3) * a.Hkv * kDim * kDim;
    const bool q_rotated = (h->L.flags & KVQ_Q_ROTATED) != 0;
    if (step) {
      step->RK = h->bank;
      step->RV = h->bank + static_cast<size_t>(a.Hkv) * kDim * kDim;
      step->mu = mu;
      step->clip_k = h->L.clip_k;
      step->clip_v = h->L.clip_v;
      step->q_rotated = q_rotated ? 1 : 0;
      e = kvq::launch_step_prep(a, *step, st);
    } else {
      e = kvq::launch_qprep(a, q_rotated ? nullptr : h->bank, mu, h->sm_scale, st);
    }
    if (e != cudaSuccess) return KVQ_ECUDA;
  }
  int slot;
  prof_begin(h, st, &slot);
  e = int2 ? kvq::launch_decode_int2(a, st) : kvq::launch_decode_bf16(a, st);
  prof_end(h, st, slot);
  if (e != cudaSuccess) return KVQ_ECUDA;
  return cuda_rc(kvq::launch_combine(a, st));
}

int append_common(kvq_handle* h, bool int2, void* pool, int num_pool_pages, const uint16_t* K,
                  const uint16_t* V, const int32_t* seq_idx, const int32_t* positions, int n,
                  const int32_t* page_table, int batch, int max_pages, void* stream) {
  if (!h || n < 0) return KVQ_EINVAL;
  if (n == 0) return KVQ_OK;
  if (!pool || !K || !V || !seq_idx || !positions || !page_table) return KVQ_EINVAL;
  if (num_pool_pages < 1 || batch < 1 || max_pages < 1) return KVQ_EINVAL;
  if (reinterpret_cast<uintptr_t>(K) % 16 || reinterpret_cast<uintptr_t>(V) % 16 ||
      reinterpret_cast<uintptr_t>(pool) % 16)
    return KVQ_EINVAL;
  if (int2 && !h->ready) return KVQ_ENOTREADY;
  kvq::DeviceGuard dev_guard(h->device);
  if (!dev_guard.ok()) return KVQ_ECUDA;
  kvq::AppendArgs a;
  a.pool = static_cast<uint8_t*>(pool);
  a.num_pool_pages = num_pool_pages;
  a.K = K;
  a.V = V;
  a.seq_idx = seq_idx;
  a.positions = positions;
  a.n = n;
  a.page_table = page_table;
  a.batch = batch;
  a.max_pages = max_pages;
  a.Hkv = h->L.num_kv_heads;
  a.R = h->bank;
  a.mu = h->bank ? h->bank + static_cast<size_t>(3) * a.Hkv * kDim * kDim : nullptr;
  a.clip_k = h->L.clip_k;
  a.clip_v = h->L.clip_v;
  a.status = h->status;
  cudaError_t e = int2 ? kvq::launch_append_int2(a, h->num_sms, S(stream))
                       : kvq::launch_append_bf16(a, S(stream));
  return cuda_rc(e);
}

}  // namespace

int kvq::handle_device(const kvq_handle* h) { return h ? h->device : -1; }

namespace {

// One thread waits on an mbarrier that nothing arrives on and no copy
// completes, with a bound of `limit_ns`: the wait runs out and the status word
// gets KVQ_STATUS_TIMEOUT, exactly as a decode or append wait that gives up.
// Nothing is in flight when the CTA leaves.
__global__ void wait_selftest_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  kvq::mbar_init(kvq::smem_u32(&bar), 1);
  kvq::fence_mbar_init();
  if (!kvq::mbar_wait_bounded(kvq::smem_u32(&bar), 0, limit_ns))
    atomicOr(status, KVQ_STATUS_TIMEOUT);
}

}  // namespace

cudaError_t kvq::launch_wait_selftest(uint32_t* status, uint64_t limit_ns, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(status, limit_ns);
  return cudaGetLastError();
}

extern "C" {

int kvq_create(const kvq_layout* layout, kvq_handle** out) {
  if (!out) return KVQ_EINVAL;
  *out = nullptr;
  if (!layout_ok(layout)) return KVQ_EINVAL;
  kvq_handle* h = new (std::nothrow) kvq_handle();
  if (!h) return KVQ_ECUDA;
  h->L = *layout;
  h->G = layout->num_heads / layout->num_kv_heads;
  h->sm_scale = layout->sm_scale > 0.f ? layout->sm_scale : 1.0f / sqrtf(static_cast<float>(kDim));
  if (cudaGetDevice(&h->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess ||
      cudaMalloc(&h->status, sizeof(uint32_t)) != cudaSuccess ||
      cudaMemset(h->status, 0, sizeof(uint32_t)) != cudaSuccess) {
    if (h->status) cudaFree(h->status);
    delete h;
    return KVQ_ECUDA;
  }
  h->ctas_int2 = kvq::decode_int2_ctas_per_sm();
  h->ctas_bf16 = kvq::decode_bf16_ctas_per_sm();
  for (int k = 0; k < 4; ++k) h->ctas_prep[k] = kvq::step_prep_ctas_per_sm(1 << k);
  *out = h;
  return KVQ_OK;
}

int kvq_destroy(kvq_handle* h) {
  if (!h) return KVQ_OK;
  kvq::DeviceGuard dev_guard(h->device);
  cudaDeviceSynchronize();
  for (int k = 0; k < kvq_handle::kSlots; ++k) {
    if (h->ev[k][0]) cudaEventDestroy(h->ev[k][0]);
    if (h->ev[k][1]) cudaEventDestroy(h->ev[k][1]);
  }
  if (h->bank) cudaFree(h->bank);
  if (h->status) cudaFree(h->status);
  delete h;
  return KVQ_OK;
}

size_t kvq_page_bytes(const kvq_handle* h) {
  return h ? static_cast<size_t>(h->L.num_kv_heads) * KVQ_INT2_RECORD_BYTES : 0;
}

size_t kvq_bf16_page_bytes(const kvq_handle* h) {
  return h ? static_cast<size_t>(h->L.num_kv_heads) * KVQ_BF16_RECORD_BYTES : 0;
}

int kvq_set_rotation(kvq_handle* h, const float* R, const float* mu, void* stream) {
  if (!h || !R || !mu) return KVQ_EINVAL;
  kvq::DeviceGuard dev_guard(h->device);
  if (!dev_guard.ok()) return KVQ_ECUDA;
  const int Hkv = h->L.num_kv_heads;
  if (!h->bank && cudaMalloc(&h->bank, rot_floats(Hkv) * sizeof(float)) != cudaSuccess) {
    h->bank = nullptr;
    return KVQ_ECUDA;
  }
  cudaStream_t st = S(stream);
  const size_t mat = static_cast<size_t>(kDim) * kDim;
  float* RVt = h->bank + 2 * Hkv * mat;
  float* mub = h->bank + 3 * Hkv * mat;
  if (cudaMemcpyAsync(h->bank, R, 2 * Hkv * mat * sizeof(float), cudaMemcpyDeviceToDevice, st) !=
          cudaSuccess ||
      cudaMemcpyAsync(mub, mu, static_cast<size_t>(Hkv) * kDim * sizeof(float),
                      cudaMemcpyDeviceToDevice, st) != cudaSuccess)
    return KVQ_ECUDA;
  if (kvq::launch_transpose(h->bank + Hkv * mat, RVt, Hkv, st) != cudaSuccess) return KVQ_ECUDA;
  h->ready = true;
  return KVQ_OK;
}

int kvq_append(kvq_handle* h, void* pool, int num_pool_pages, const uint16_t* K,
               const uint16_t* V, const int32_t* seq_idx, const int32_t* positions, int n,
               const int32_t* page_table, int batch, int max_pages, void* stream) {
  return append_common(h, true, pool, num_pool_pages, K, V, seq_idx, positions, n, page_table,
                       batch, max_pages, stream);
}

int kvq_bf16_append(kvq_handle* h, void* pool, int num_pool_pages, const uint16_t* K,
                    const uint16_t* V, const int32_t* seq_idx, const int32_t* positions, int n,
                    const int32_t* page_table, int batch, int max_pages, void* stream) {
  return append_common(h, false, pool, num_pool_pages, K, V, seq_idx, positions, n, page_table,
                       batch, max_pages, stream);
}

size_t kvq_workspace_bytes(const kvq_handle* h, int batch, int num_splits) {
  if (!h || batch < 1 || num_splits < 0 || num_splits > kvq::kMaxSplits) return 0;
  const int s = num_splits ? num_splits : splits_cap(h, batch, true);
  return kvq::decode_ws_layout(batch, h->L.num_kv_heads, h->L.num_heads, s, true).total;
}

size_t kvq_bf16_workspace_bytes(const kvq_handle* h, int batch, int num_splits) {
  if (!h || batch < 1 || num_splits < 0 || num_splits > kvq::kMaxSplits) return 0;
  const int s = num_splits ? num_splits : splits_cap(h, batch, false);
  return kvq::decode_ws_layout(batch, h->L.num_kv_heads, h->L.num_heads, s, false).total;
}

int kvq_auto_splits(const kvq_handle* h, int batch, int max_pages) {
  if (!h || batch < 1 || max_pages < 1) return 0;
  return choose_splits(h, batch, max_pages, true);
}

int kvq_decode(kvq_handle* h, const void* pool, int num_pool_pages, const uint16_t* q,
               const int32_t* page_table, int max_pages, const int32_t* seq_lens, int batch,
               float* out, void* workspace, size_t ws_bytes, int num_splits, void* stream) {
  return decode_common(h, true, pool, num_pool_pages, q, page_table, max_pages, seq_lens, batch,
                       out, workspace, ws_bytes, num_splits, stream);
}

int kvq_decode_window(kvq_handle* h, const void* pool, int num_pool_pages,
                      const void* bf16_pool, int bf16_num_pool_pages,
                      const int32_t* bf16_page_table, const uint16_t* q,
                      const int32_t* page_table, int max_pages, const int32_t* seq_lens, int batch,
                      int sink, int recent, float* out, void* workspace, size_t ws_bytes,
                      int num_splits, void* stream) {
  Window win;
  win.bf16_pool = bf16_pool;
  win.bf16_num_pool_pages = bf16_num_pool_pages;
  win.bf16_page_table = bf16_page_table;
  win.sink = sink;
  win.recent = recent;
  win.on = true;
  return decode_common(h, true, pool, num_pool_pages, q, page_table, max_pages, seq_lens, batch,
                       out, workspace, ws_bytes, num_splits, stream, win);
}

int kvq_append_decode(kvq_handle* h, void* pool, int num_pool_pages, const uint16_t* K_new,
                      const uint16_t* V_new, const uint16_t* q, const int32_t* page_table,
                      int max_pages, const int32_t* seq_lens, int batch, float* out,
                      void* workspace, size_t ws_bytes, int num_splits, void* stream) {
  if (!K_new || !V_new) return KVQ_EINVAL;
  if (reinterpret_cast<uintptr_t>(K_new) % 4 || reinterpret_cast<uintptr_t>(V_new) % 4)
    return KVQ_EINVAL;
  kvq::StepArgs step;
  step.pool = static_cast<uint8_t*>(pool);
  step.K = K_new;
  step.V = V_new;
  return decode_common(h, true, pool, num_pool_pages, q, page_table, max_pages, seq_lens, batch,
                       out, workspace, ws_bytes, num_splits, stream, Window(), &step);
}

int kvq_append_decode_window(kvq_handle* h, void* pool, int num_pool_pages, void* bf16_pool,
                             int bf16_num_pool_pages, const int32_t* bf16_page_table,
                             const uint16_t* K_new, const uint16_t* V_new, const uint16_t* q,
                             const int32_t* page_table, int max_pages, const int32_t* seq_lens,
                             int batch, int sink, int recent, float* out, void* workspace,
                             size_t ws_bytes, int num_splits, void* stream) {
  if (!K_new || !V_new) return KVQ_EINVAL;
  if (reinterpret_cast<uintptr_t>(K_new) % 4 || reinterpret_cast<uintptr_t>(V_new) % 4)
    return KVQ_EINVAL;
  Window win;
  win.bf16_pool = bf16_pool;
  win.bf16_num_pool_pages = bf16_num_pool_pages;
  win.bf16_page_table = bf16_page_table;
  win.sink = sink;
  win.recent = recent;
  win.on = true;
  kvq::StepArgs step;
  step.pool = static_cast<uint8_t*>(pool);
  step.K = K_new;
  step.V = V_new;
  step.bf16_pool = static_cast<uint8_t*>(bf16_pool);
  step.bf16_num_pool_pages = bf16_num_pool_pages;
  step.bf16_page_table = bf16_page_table;
  return decode_common(h, true, pool, num_pool_pages, q, page_table, max_pages, seq_lens, batch,
                       out, workspace, ws_bytes, num_splits, stream, win, &step);
}

int kvq_bf16_decode(kvq_handle* h, const void* pool, int num_pool_pages, const uint16_t* q,
                    const int32_t* page_table, int max_pages, const int32_t* seq_lens, int batch,
                    float* out, void* workspace, size_t ws_bytes, int num_splits, void* stream) {
  if (h && num_splits == 0) num_splits = choose_splits(h, batch, max_pages, false);
  return decode_common(h, false, pool, num_pool_pages, q, page_table, max_pages, seq_lens, batch,
                       out, workspace, ws_bytes, num_splits, stream);
}

int kvq_dequant(kvq_handle* h, const void* pool, int num_pool_pages, const int32_t* page_table,
                int max_pages, int seq, int start, int len, float* K_out, float* V_out,
                void* stream) {
  if (!h || !pool || !page_table || len < 0 || seq < 0 || start < 0) return KVQ_EINVAL;
  if (num_pool_pages < 1 || max_pages < 1) return KVQ_EINVAL;
  if (len == 0 || (!K_out && !V_out)) return KVQ_OK;
  kvq::DeviceGuard dev_guard(h->device);
  if (!dev_guard.ok()) return KVQ_ECUDA;
  return cuda_rc(kvq::launch_dequant(static_cast<const uint8_t*>(pool), num_pool_pages,
                                     page_table, max_pages, h->L.num_kv_heads, seq, start, len,
                                     K_out, V_out, h->status, S(stream)));
}

int kvq_get_status(kvq_handle* h, uint32_t* bits, void* stream) {
  if (!h || !bits) return KVQ_EINVAL;
  kvq::DeviceGuard dev_guard(h->device);
  if (!dev_guard.ok()) return KVQ_ECUDA;
  cudaStream_t st = S(stream);
  uint32_t v = 0;
  if (cudaMemcpyAsync(&v, h->status, sizeof(uint32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
      cudaMemsetAsync(h->status, 0, sizeof(uint32_t), st) != cudaSuccess ||
      cudaStreamSynchronize(st) != cudaSuccess)
    return KVQ_ECUDA;
  *bits = v;
  return KVQ_OK;
}

int kvq_selftest_wait_timeout(kvq_handle* h, int limit_us, void* stream) {
  if (!h || limit_us < 1 || limit_us > 1000000) return KVQ_EINVAL;
  kvq::DeviceGuard dev_guard(h->device);
  if (!dev_guard.ok()) return KVQ_ECUDA;
  return cuda_rc(kvq::launch_wait_selftest(h->status, 1000ull * static_cast<uint64_t>(limit_us),
                                           S(stream)));
}

int kvq_profile_enable(kvq_handle* h, int enable) {
  if (!h) return KVQ_EINVAL;
  h->prof = enable != 0;
  h->total_ms = 0.0;
  h->launches = 0;
  for (int k = 0; k < kvq_handle::kSlots; ++k) h->pending[k] = false;
  h->next = 0;
  return KVQ_OK;
}

int kvq_profile_read(kvq_handle* h, double* total_ms, int* launches) {
  if (!h || !total_ms || !launches) return KVQ_EINVAL;
  for (int k = 0; k < kvq_handle::kSlots; ++k) {
    if (!h->pending[k]) continue;
    float ms = 0.f;
    if (cudaEventSynchronize(h->ev[k][1]) != cudaSuccess ||
        cudaEventElapsedTime(&ms, h->ev[k][0], h->ev[k][1]) != cudaSuccess)
      return KVQ_ECUDA;
    h->total_ms += ms;
    h->pending[k] = false;
  }
  *total_ms = h->total_ms;
  *launches = h->launches;
  h->total_ms = 0.0;
  h->launches = 0;
  h->next = 0;
  return KVQ_OK;
}

namespace {
bool optr_shape_ok(int Hkv, int T, int Nq, int G, int Dm) {
  return Hkv >= 1 && Hkv <= 64 && Nq >= 1 && T >= Nq && T <= (1 << 20) && G >= 1 && G <= 8 &&
         Dm >= 1 && Dm <= 65536 && static_cast<long long>(Nq) * G <= 65535;
}
}  // namespace

size_t kvq_optr_workspace_bytes(int num_kv_heads, int T, int Nq, int G, int Dm) {
  if (!optr_shape_ok(num_kv_heads, T, Nq, G, Dm)) return 0;
  return kvq::optr_workspace_bytes(num_kv_heads, T, Nq, G, Dm);
}

int kvq_optr_calibrate(int num_kv_heads, int T, int Nq, int G, int Dm, const uint16_t* K,
                       const uint16_t* V, const uint16_t* Q, const float* W_O, const float* R0,
                       const float* mu, float clip_k, float clip_v, float lambda_k, float lr,
                       int steps, float sm_scale, float* R_out, float* history, void* workspace,
                       size_t ws_bytes, void* stream) {
  if (!optr_shape_ok(num_kv_heads, T, Nq, G, Dm)) return KVQ_EINVAL;
  if (!K || !V || !Q || !W_O || !R0 || !mu || !R_out || !history || !workspace) return KVQ_EINVAL;
  if (!(clip_k > 0.f && clip_k <= 1.f) || !(clip_v > 0.f && clip_v <= 1.f)) return KVQ_EINVAL;
  if (!(lr > 0.f) || !(lambda_k >= 0.f) || steps < 0 || steps > 100000) return KVQ_EINVAL;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return KVQ_EINVAL;
  if (ws_bytes < kvq::optr_workspace_bytes(num_kv_heads, T, Nq, G, Dm)) return KVQ_ENOSPACE;
  const float scale = sm_scale > 0.f ? sm_scale : 1.0f / sqrtf(static_cast<float>(kDim));
  return kvq::optr_calibrate(num_kv_heads, T, Nq, G, Dm, K, V, Q, W_O, R0, mu, clip_k, clip_v,
                             lambda_k, lr, steps, scale, R_out, history, workspace, S(stream));
}

int kvq_optr_loss_grad(int num_kv_heads, int T, int Nq, int G, int Dm, const uint16_t* K,
                       const uint16_t* V, const uint16_t* Q, const float* W_O, const float* R0,
                       const float* mu, float clip_k, float clip_v, float lambda_k,
                       float sm_scale, const float* A_key, const float* A_value, int which,
                       float* loss, float* grad, void* workspace, size_t ws_bytes, void* stream) {
  if (!optr_shape_ok(num_kv_heads, T, Nq, G, Dm)) return KVQ_EINVAL;
  if (!K || !V || !Q || !W_O || !R0 || !mu || !A_key || !loss || !grad || !workspace)
    return KVQ_EINVAL;
  if (which != 0 && which != 1) return KVQ_EINVAL;
  if (which == 1 && !A_value) return KVQ_EINVAL;
  if (!(clip_k > 0.f && clip_k <= 1.f) || !(clip_v > 0.f && clip_v <= 1.f)) return KVQ_EINVAL;
  if (!(lambda_k >= 0.f)) return KVQ_EINVAL;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return KVQ_EINVAL;
  if (ws_bytes < kvq::optr_workspace_bytes(num_kv_heads, T, Nq, G, Dm)) return KVQ_ENOSPACE;
  const float scale = sm_scale > 0.f ? sm_scale : 1.0f / sqrtf(static_cast<float>(kDim));
  return kvq::optr_loss_grad(num_kv_heads, T, Nq, G, Dm, K, V, Q, W_O, R0, mu, clip_k, clip_v,
                             lambda_k, scale, A_key, A_value, which, loss, grad, workspace,
                             S(stream));
}

const char* kvq_strerror(int code) {
  switch (code) {
    case KVQ_OK: return "ok";
    case KVQ_EINVAL: return "invalid argument or unsupported layout";
    case KVQ_ENOSPACE: return "workspace too small";
    case KVQ_ECUDA: return "CUDA runtime error or kernel launch failure";
    case KVQ_ENOTREADY: return "rotation bank not set (call kvq_set_rotation first)";
    default: return "unknown kvq error code";
  }
}

}  // extern "C"
