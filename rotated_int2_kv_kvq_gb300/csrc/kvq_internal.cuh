// kvq_internal.cuh — shared declarations of the CUDA side of libkvq (sm_103a).
//
// Nothing here is part of the public ABI (include/kvq.h).
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "kvq.h"

namespace kvq {

constexpr int kDim = 128;          // head_dim
constexpr int kPage = 16;          // tokens per page
constexpr int kInt2Rec = KVQ_INT2_RECORD_BYTES;   // bytes per (page, kv head)
constexpr int kBf16Rec = KVQ_BF16_RECORD_BYTES;
constexpr int kMaxG = 4;           // query heads per KV head handled per CTA
constexpr int kPartStride = 132;   // floats per split partial: m, l, 2 pad, o[128]
constexpr int kQFragWords = 32 * 16;   // uint32 per (b, kv): 32 lanes x 16 B-fragment regs
constexpr int kQMeta = 12;         // floats per (b, kv): {kappa, zeta} x 4 heads, q.mu x 4 heads
constexpr int kMaxSplits = 1024;
constexpr int kDecodeWarps = 4;    // BF16 decode CTA
constexpr int kInt2Warps = 8;      // INT2 decode CTA
constexpr int kDecodeThreads = kDecodeWarps * 32;

// Workspace layout of one decode call (offsets in bytes, each 256-aligned).
struct DecodeWs {
  size_t qfrag_off, qmeta_off, part_off, sched_off, total;
};
DecodeWs decode_ws_layout(int batch, int Hkv, int H, int splits, bool int2);

struct DecodeArgs {
  const uint8_t* pool;
  int num_pool_pages;
  const uint16_t* q;
  const int32_t* page_table;
  int max_pages;
  const int32_t* seq_lens;
  int batch;
  int H, Hkv, G;
  int splits, chunk_pages;
  int hpc;                   // KV heads per INT2 decode CTA (1, 2, 4 or 8; divides Hkv)
  const uint32_t* qfrag;     // [B][Hkv][32][16]
  const float* qmeta;        // [B][Hkv][kQMeta]: kappa, zeta per head, then q.mu per head
  float* part;               // [B][H][splits][kPartStride]
  float* out;                // [B][H][D]
  const float* RVt;          // [Hkv][D][D] transposed value rotations
  const float* RV;           // [Hkv][D][D] value rotations
  int rotate_out;            // 1: out = o_rot R_V^T, 0: out = o_rot
  int combine_per_head = 0;  // 1: the combine takes one CTA per query head (no window)
  int combine_small = 0;     // 1: the KV-head combine runs in 256-thread CTAs, four per SM (large batches)
  // Length-balanced schedule (balanced = 1): the decode grid's batch * splits
  // CTAs are shared out over the sequences in chunks of one common size, in
  // proportion to their page counts.  sched_map[c] = {b, chunk index, first
  // partial slot of b, chunk pages} of CTA c (b = -1: no chunk); sequence b's
  // partials sit in slots sched_base[b] .. sched_base[b] + sched_nsplit[b] - 1,
  // partial (slot, head) at part[(slot * H + head) * kPartStride].  The table
  // is written by an extra CTA of the query-preparation kernel.
  int prep_nb = 1;            // sequences per step-preparation append CTA (1, 2, 4, 8); query CTAs take min(prep_nb, 2)
  int balanced = 0;
  int sched_ctas = 0;          // chunks the balanced schedule may use: whole waves of CTAs
  int4* sched_map = nullptr;   // [batch * splits]
  int* sched_nsplit = nullptr; // [batch]
  int* sched_base = nullptr;   // [batch]
  uint32_t* status;
  float log2_scale;          // sm_scale * log2(e)
  // BF16 window (sink + recent tokens); window = 0 for a plain decode
  int window;
  int win_sink, win_recent;
  const uint8_t* bf16_pool;
  int bf16_num_pool_pages;
  const int32_t* bf16_page_table;   // [B][max_pages]
};

struct AppendArgs {
  uint8_t* pool;
  int num_pool_pages;
  const uint16_t* K;
  const uint16_t* V;
  const int32_t* seq_idx;
  const int32_t* positions;
  int n;
  const int32_t* page_table;
  int batch, max_pages, Hkv;
  const float* R;            // [2][Hkv][D][D]
  const float* mu;           // [Hkv][D]
  float clip_k, clip_v;
  uint32_t* status;
};

// The append half of kvq_append_decode: one new token per sequence.
struct StepArgs {
  uint8_t* pool;
  const uint16_t* K;         // [B][Hkv][D] bf16, the token at position seq_lens[b] - 1
  const uint16_t* V;
  const float* RK;           // [Hkv][D][D]
  const float* RV;           // [Hkv][D][D]
  const float* mu;           // [Hkv][D]
  float clip_k, clip_v;
  int q_rotated;             // 1: q is already q R_K
  // BF16 window cache: the token is also copied there (kvq_append_decode_window);
  // bf16_pool == nullptr for kvq_append_decode
  uint8_t* bf16_pool = nullptr;
  int bf16_num_pool_pages = 0;
  const int32_t* bf16_page_table = nullptr;
};

// ---- launchers (defined in the .cu files) --------------------------------
cudaError_t launch_append_int2(const AppendArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_append_bf16(const AppendArgs& a, cudaStream_t st);
cudaError_t launch_qprep(const DecodeArgs& a, const float* RK, const float* mu, float sm_scale,
                         cudaStream_t st);
cudaError_t launch_step_prep(const DecodeArgs& a, const StepArgs& sa, cudaStream_t st);
cudaError_t launch_decode_int2(const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_decode_bf16(const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_combine(const DecodeArgs& a, cudaStream_t st);
cudaError_t launch_dequant(const uint8_t* pool, int num_pool_pages, const int32_t* page_table,
                           int max_pages, int Hkv, int seq, int start, int len, float* K_out,
                           float* V_out, uint32_t* status, cudaStream_t st);
cudaError_t launch_transpose(const float* in, float* out, int count, cudaStream_t st);
size_t optr_workspace_bytes(int H, int T, int Nq, int G, int Dm);
int optr_calibrate(int H, int T, int Nq, int G, int Dm, const uint16_t* K, const uint16_t* V,
                   const uint16_t* Q, const float* W, const float* R0, const float* mu,
                   float clip_k, float clip_v, float lambda_k, float lr, int steps, float sm_scale,
                   float* R_out, float* hist, void* workspace, cudaStream_t st);
int optr_loss_grad(int H, int T, int Nq, int G, int Dm, const uint16_t* K, const uint16_t* V,
                   const uint16_t* Q, const float* W, const float* R0, const float* mu,
                   float clip_k, float clip_v, float lambda_k, float sm_scale, const float* A_key,
                   const float* A_value, int which, float* loss, float* grad, void* workspace,
                   cudaStream_t st);
int decode_int2_ctas_per_sm();
int combine_head_ctas_per_sm();
int step_prep_ctas_per_sm(int nb);  // nb = 1, 2, 4 or 8 sequences per CTA
int decode_bf16_ctas_per_sm();
// Makes `dev` the calling thread's current device while the guard lives and
// gives the caller's device back afterwards, so that no entry point changes
// the caller's current device.
class DeviceGuard {
 public:
  explicit DeviceGuard(int dev) {
    ok_ = cudaGetDevice(&prev_) == cudaSuccess;
    if (ok_ && prev_ != dev) {
      ok_ = cudaSetDevice(dev) == cudaSuccess;
      changed_ = ok_;
    }
  }
  ~DeviceGuard() {
    if (changed_) cudaSetDevice(prev_);
  }
  DeviceGuard(const DeviceGuard&) = delete;
  DeviceGuard& operator=(const DeviceGuard&) = delete;
  bool ok() const { return ok_; }

 private:
  int prev_ = 0;
  bool ok_ = false, changed_ = false;
};

int handle_device(const kvq_handle* h);   // CUDA device the handle was created on
cudaError_t launch_wait_selftest(uint32_t* status, uint64_t limit_ns, cudaStream_t st);

// ---- device helpers -------------------------------------------------------
#if defined(__CUDACC__)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// One attempt that lets the thread sleep (up to `ns` nanoseconds) until the
// phase completes instead of returning at once.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Nanoseconds of the GPU's global timer.
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Default bound of every wait on a page copy: two seconds.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Wait for phase `parity` of an mbarrier, giving up once `limit_ns` of global
// time have passed (returns false; the caller records KVQ_STATUS_TIMEOUT).
// Each attempt lets the thread sleep up to 0.1 ms until the phase completes.
// The attempt count is capped too (2^29 attempts, far beyond any limit used
// here), so the wait ends even if the timer did not advance.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0; it < (1u << 26); ++it) {
    for (int i = 0; i < 8; ++i)
      if (mbar_try_wait_sleep(bar, parity, 100000u)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
  return false;
}

// After a bounded wait on phase `parity` of `bar` gave up: wait once more
// (bounded) so that a copy still in flight into this CTA's shared memory lands
// before the CTA can exit and its shared memory be given to another CTA.
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
  (void)mbar_wait_bounded(bar, parity);
}

// One-dimensional bulk copy global -> shared (TMA, no tensor map), completing
// `bytes` of transaction count on `bar`.  dst, src 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Transpose of an 8 x 8 matrix of 16-bit elements held in mma fragment order
// (lane (g, t) holds row g, columns 2t and 2t+1): lane (g, t) receives column
// g, rows 2t and 2t+1.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 2^x via the SFU (ex2.approx.ftz): 2^-inf = 0, 2^0 = 1.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// log2(x) via the SFU (lg2.approx.ftz): log2(0) = -inf.
__device__ __forceinline__ float fast_log2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float half_lo(uint32_t h2) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xffffu)));
}
__device__ __forceinline__ float half_hi(uint32_t h2) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf162(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

#endif  // __CUDACC__

}  // namespace kvq
