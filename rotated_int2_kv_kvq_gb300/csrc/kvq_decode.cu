// kvq_decode.cu — split-K decode attention over the paged INT2 cache (and the
// BF16 comparison cache), the log-sum-exp combine with the inverse value
// rotation, and the dequantisation test export.
//
// Method: "Output-Aware Rotation for INT2 KV-Cache Quantization" (pith.science
// review of arXiv 2608.02691).  Decode reads the rotated, centred, quantised
// keys with the rotated query (rotation is orthogonal, "What carries the
// argument" mechanism 1; centring only shifts every logit by q.mu, mechanism 2),
// and reads values back with dequantisation and the inverse rotation (mechanism
// 3), which deployment may fold into W_V / W_O ("If this is right", third item).
// Split-K with a log-sum-exp merge follows the FlashDecoding scheme named as
// the comparison point on "The KV cache goes on a diet", "Crush it to INT2".
//
// How the INT2 kernel maps onto sm_103a
// -------------------------------------
// One CTA = 8 warps = one (split, group of HPC KV heads, sequence); warp w
// serves KV head w / (8/HPC) of the group and takes every (8/HPC)-th page of
// the split.  Each warp streams its own pages through its own ring of stages:
// lane 0 issues 1-D TMA bulk copies (cp.async.bulk, mbarrier completion) of the
// head's 1152-byte records, four pages per stage and two stages per warp, and
// refills a stage as soon as the warp has read it.  The warp takes a stage's
// pages in pairs (two independent tensor-core chains in flight).  No
// stage is shared between warps, so a warp that runs ahead never waits for a
// slower one (sharing one copy of a page between the CTA's heads made every
// warp keep the pace of the slowest and cost 6 %).  A page record holds the 16
// tokens' codes in tensor-core fragment order, so each lane takes its share of
// a page with one 16-byte shared load and hands it to mma.sync.m16n8k16 without shuffling:
//   scores  S[token][col] = Kcode[token][dim] . B[dim][col]     (M = 16 tokens)
//   values  O^T[dim][col] += Vcode^T[dim][token] . P[token][col] (M = 16 dims)
// with col = 2*head + {hi, lo}: each operand that is not a code is split into an
// fp16 high part and an fp16 residual (the query's scaled by 2^11 so it stays a
// normal number), which keeps products at fp32 accuracy.  Codes become fp16 operands
// with one AND each (and one or two shifts per word of 16 codes): a 2-bit field
// at bit offset B < 9 of a 16-bit half is the fp16 number code * 2^(B - 24),
// exactly; the powers of two are folded into the query operands and removed in
// the value epilogue.
//
// Kernel chain of one decode call: qprep (or step_prep, which also appends the
// new token) -> decode -> combine, each launched as a programmatic dependent of
// the previous kernel (griddepcontrol), so each one is resident and waiting when
// its predecessor finishes.
#include "kvq_internal.cuh"

#include <math.h>


namespace kvq {

DecodeWs decode_ws_layout(int batch, int Hkv, int H, int splits, bool int2) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  DecodeWs w;
  size_t o = 0;
  w.qfrag_off = o;
  if (int2) o += up(static_cast<size_t>(batch) * Hkv * kQFragWords * 4);
  w.qmeta_off = o;
  if (int2) o += up(static_cast<size_t>(batch) * Hkv * kQMeta * 4);
  w.part_off = o;
  o += up(static_cast<size_t>(batch) * H * splits * kPartStride * 4);
  w.sched_off = o;
  if (int2) o += up(static_cast<size_t>(batch) * splits * 16 + static_cast<size_t>(batch) * 8);
  w.total = o;
  return w;
}

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kStagesBf16 = 3;

// Programmatic dependent launch (no-ops when the kernel is launched normally).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Bit offset, within its fp16 half, of the tensor-core operand made from code
// position P (0..7) of a fragment word (see field_op below): the operand is
// code * 2^(code_bit(P) - 24).
__host__ __device__ constexpr int code_bit(int P) { return P < 2 ? 2 * P + 6 : (P < 5 ? 2 * P : 2 * P - 6); }

// ---------------------------------------------------------------------------
// Query preparation: q_rot = q R_K for the G query heads of one sequence and one
// KV head per CTA (R_K staged in shared memory by a bulk copy), then the
// scores' B fragments.  B[row][col] for k-block w holds x = q_rot[head][16w+row]
// * 2^(e_head + 8 - code_bit(w)), where 2^e_head brings max|q_rot| into
// [2^10, 2^11) (so x < 2^15 stays an fp16 number): column 2*head is fp16(x),
// column 2*head+1 the residual (x - fp16(x)) * 2^11.  Codes of k-block w enter
// as code * 2^(code_bit(w) - 24), so every product is code * q_rot * 2^(e - 16)
// and the score of a token is q_rot . c = 2^(16 - e) * (hi + 2^-11 lo).  Per head also: kappa =
// sm_scale*log2e * 2^(16 - e), zeta = sm_scale*log2e * sum(q_rot) and
// qmu = sm_scale*log2e * (q . mu), the logit shift that centring the keys took
// out ("What carries the argument", mechanism 2); only a decode that mixes INT2
// and BF16 tokens in one softmax needs it back.
// RK == nullptr: q is already rotated (KVQ_Q_ROTATED) and is used as it is.
// Launched as a programmatic dependent of the preceding kernel: the bulk copy
// of R_K (set by kvq_set_rotation, complete before any decode call starts) is
// issued before the kernel waits for its predecessor; q, which a preceding
// kernel may still be writing, is read only after that wait.
// ---------------------------------------------------------------------------
template <int NB>
struct QprepSmem {
  float R[kDim * kDim];
  float qs[NB][kMaxG][kDim];
  float qr[NB][kMaxG][kDim];
  int e[kMaxG];
  uint64_t bar;
};

// Second half of the query preparation, shared by qprep_kernel and
// step_prep_kernel (128 threads, called by all of them once qr is complete):
// per-head sum, max|.| and q.mu, the logit constants, and the B fragments.
__device__ __forceinline__ void qprep_tail(const DecodeArgs& a, float (&qs)[kMaxG][kDim],
                                           float (&qr)[kMaxG][kDim], int (&e_sm)[kMaxG],
                                           const float* __restrict__ mu, float log2_scale, int b,
                                           int kv) {
  const int i = threadIdx.x, G = a.G;
  // per-vector sum and max|.|: warp w handles vector w
  {
    const int w = i >> 5, lane = i & 31;
    float s = 0.0f, m = 0.0f, qm = 0.0f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float x = qr[w][lane + 32 * k];
      s += x;
      m = fmaxf(m, fabsf(x));
      qm = fmaf(qs[w][lane + 32 * k], mu[static_cast<size_t>(kv) * kDim + lane + 32 * k], qm);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      s += __shfl_xor_sync(0xffffffffu, s, off);
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      qm += __shfl_xor_sync(0xffffffffu, qm, off);
    }
    if (lane == 0) {
      int e = 0;
      if (m > 0.0f && m < INFINITY) {
        int E;
        frexpf(m, &E);           // m = f * 2^E, f in [0.5, 1)
        e = 11 - E;              // m * 2^e in [2^10, 2^11)
      }
      e_sm[w] = e;
      float* meta = const_cast<float*>(a.qmeta) + (static_cast<size_t>(b) * a.Hkv + kv) * kQMeta;
      meta[2 * w] = (w < G) ? log2_scale * ldexpf(1.0f, 16 - e) : 0.0f;
      meta[2 * w + 1] = (w < G) ? log2_scale * s : 0.0f;
      meta[8 + w] = (w < G) ? log2_scale * qm : 0.0f;
    }
  }
  __syncthreads();
  // B fragments: 32 lanes x 16 registers; thread i writes 4 registers of lane i/4
  {
    const int L = i >> 2, quad = i & 3;
    const int g = L >> 2, t = L & 3, head = g >> 1, part = g & 1;
    uint32_t out[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int r = 4 * quad + k;
      const int w = r >> 1, which = r & 1;
      const int row = 16 * w + 2 * t + 8 * which;
      float x2[2] = {0.0f, 0.0f};
      if (head < G) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          // codes of k-block w enter as c * 2^(code_bit(w) - 24): every
          // product is c * q * 2^(e - 16)
          const float x = ldexpf(qr[head][row + u], e_sm[head] + 8 - code_bit(w));
          const __half hi = __float2half_rn(x);
          x2[u] = part ? (x - __half2float(hi)) * 2048.0f : __half2float(hi);
        }
      }
      out[k] = pack_half2(x2[0], x2[1]);
    }
    uint32_t* dst = const_cast<uint32_t*>(a.qfrag) +
                    ((static_cast<size_t>(b) * a.Hkv + kv) * 32 + L) * 16 + 4 * quad;
    *reinterpret_cast<uint4*>(dst) = make_uint4(out[0], out[1], out[2], out[3]);
  }
}

// One CTA per (group of NB sequences, KV head): R_K is staged once; thread i
// computes element i of the G rotated query vectors of each sequence, one fmaf
// chain over j = 0..127 each (the chains of the group's sequences side by
// side), with the query elements read four j at a time (one broadcast load per
// vector).  Sequences b0 .. b0 + nb - 1 (nb <= NB) are prepared.
template <int NB>
__device__ __forceinline__ void qprep_cta(const DecodeArgs& a, const float* __restrict__ RK,
                                          const float* __restrict__ mu, float log2_scale,
                                          QprepSmem<NB>& sm, int b0, int nb, int kv) {
  const int i = threadIdx.x;
  const int G = a.G;
  const bool rotate = RK != nullptr;
  const uint32_t bar = smem_u32(&sm.bar);
  if (rotate && i == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, kDim * kDim * 4);
    bulk_g2s(smem_u32(sm.R), RK + static_cast<size_t>(kv) * kDim * kDim, kDim * kDim * 4, bar);
  }
  __syncthreads();     // the barrier is initialised before any thread waits on it
  griddep_wait();      // q may come from the preceding kernel
#pragma unroll
  for (int u = 0; u < NB; ++u)
#pragma unroll
    for (int h = 0; h < kMaxG; ++h) {
      float x = 0.0f;
      if (h < G && u < nb) {
        const uint16_t bits = a.q[(static_cast<size_t>(b0 + u) * a.H + kv * G + h) * kDim + i];
        x = __uint_as_float(static_cast<uint32_t>(bits) << 16);
      }
      sm.qs[u][h][i] = x;
    }
  if (rotate) {
    const bool ok = mbar_wait_bounded(bar, 0);
    if (__syncthreads_or(!ok)) {
      if (i == 0) {
        atomicOr(a.status, KVQ_STATUS_TIMEOUT);
        mbar_drain(bar, 0);
      }
      return;
    }
    float acc[NB][kMaxG];
#pragma unroll
    for (int u = 0; u < NB; ++u)
#pragma unroll
      for (int h = 0; h < kMaxG; ++h) acc[u][h] = 0.0f;
#pragma unroll 2
    for (int j0 = 0; j0 < kDim; j0 += 4) {
      float r[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) r[k] = sm.R[(j0 + k) * kDim + i];
#pragma unroll
      for (int u = 0; u < NB; ++u)
#pragma unroll
        for (int h = 0; h < kMaxG; ++h) {
          const float4 x = *reinterpret_cast<const float4*>(&sm.qs[u][h][j0]);
          acc[u][h] = fmaf(x.x, r[0], acc[u][h]);
          acc[u][h] = fmaf(x.y, r[1], acc[u][h]);
          acc[u][h] = fmaf(x.z, r[2], acc[u][h]);
          acc[u][h] = fmaf(x.w, r[3], acc[u][h]);
        }
    }
#pragma unroll
    for (int u = 0; u < NB; ++u)
#pragma unroll
      for (int h = 0; h < kMaxG; ++h) sm.qr[u][h][i] = acc[u][h];
  } else {
#pragma unroll
    for (int u = 0; u < NB; ++u)
#pragma unroll
      for (int h = 0; h < kMaxG; ++h) sm.qr[u][h][i] = sm.qs[u][h][i];
  }
  __syncthreads();
  for (int u = 0; u < nb; ++u) {
    if (u > 0) __syncthreads();        // sm.e of the previous sequence has been read
    qprep_tail(a, sm.qs[u], sm.qr[u], sm.e, mu, log2_scale, b0 + u, kv);
  }
}

// ---------------------------------------------------------------------------
// Length-balanced decode schedule (a.balanced), written by one extra CTA of
// the query-preparation kernel (128 threads) after its dependency wait: the
// smallest chunk size P (pages) such that the batch's chunks, ceil(n_b / P) for
// a sequence of n_b pages, number at most a.sched_ctas (whole waves of the
// decode grid's batch * splits CTAs) and
// at most kMaxSplits per sequence, and at least 8 pages unless no sequence is
// that long; then each sequence's chunk count, the first partial slot of each
// sequence (prefix sum) and the CTA -> (sequence, chunk) map.  A sequence with
// an invalid length gets no chunk (its output is 0) and sets
// KVQ_STATUS_BAD_SEQLEN.  With equal lengths the chunks are those of the plain
// schedule (the same split count per sequence).
// ---------------------------------------------------------------------------
__device__ __forceinline__ int block_sum128(int v, int* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  __syncthreads();                       // red may still be read from a previous call
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  return (red[0] + red[1]) + (red[2] + red[3]);
}

// nsm: the kernel's (otherwise unused) dynamic shared memory, nsm_len ints:
// the page counts live there when the batch fits, else in sched_nsplit.
__device__ void schedule_cta(const DecodeArgs& a, int* nsm, int nsm_len) {
  __shared__ int red[4];
  __shared__ int scan[128];
  const int tid = threadIdx.x, B = a.batch;
  const int C = a.batch * a.splits;            // decode CTAs along x (map entries)
  const int Cuse = min(C, a.sched_ctas);        // chunks used: whole waves of CTAs
  griddep_wait();                              // seq_lens may come from a predecessor
  // pages of each sequence, kept in shared memory (or sched_nsplit) until the
  // chunk size is known
  int* const np = B <= nsm_len ? nsm : a.sched_nsplit;
  int nmax = 0;
  for (int b = tid; b < B; b += 128) {
    const int len = a.seq_lens[b];
    int n = 0;
    if (len < 0 || len > a.max_pages * kPage) atomicOr(a.status, KVQ_STATUS_BAD_SEQLEN);
    else n = (len + kPage - 1) / kPage;
    np[b] = n;
    nmax = max(nmax, n);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) nmax = max(nmax, __shfl_xor_sync(0xffffffffu, nmax, off));
  if ((tid & 31) == 0) red[tid >> 5] = nmax;
  __syncthreads();
  nmax = max(max(red[0], red[1]), max(red[2], red[3]));
  // smallest P in [1, max(nmax, 1)] with sum_b ceil(n_b / P) <= C and
  // ceil(nmax / P) <= kMaxSplits (P = nmax always qualifies: one chunk each)
  int lo = 1, hi = max(nmax, 1);
  while (lo < hi) {                            // uniform across the CTA
    const int P = (lo + hi) >> 1;
    int cnt = 0;
    for (int b = tid; b < B; b += 128) cnt += (np[b] + P - 1) / P;
    cnt = block_sum128(cnt, red);
    if (cnt <= Cuse && (nmax + P - 1) / P <= kMaxSplits) hi = P;
    else lo = P + 1;
  }
  const int P = max(lo, min(8, max(nmax, 1)));
  // chunk counts and their exclusive prefix: thread t takes sequences
  // [t * per, (t + 1) * per)
  const int per = (B + 127) / 128;
  const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
  int local = 0;
  for (int b = b0; b < b1; ++b) local += (np[b] + P - 1) / P;
  scan[tid] = local;
  __syncthreads();
  if (tid < 32) {                              // warp 0 scans the 128 partial sums
    int v[4], sum = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) { v[k] = scan[4 * tid + k]; sum += v[k]; }
    int x = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (tid >= off) x += y;
    }
    int run = x - sum;                         // exclusive prefix of this lane's four
#pragma unroll
    for (int k = 0; k < 4; ++k) { scan[4 * tid + k] = run; run += v[k]; }
  }
  __syncthreads();
  int base = scan[tid];
  for (int b = b0; b < b1; ++b) {
    const int ns = (np[b] + P - 1) / P;
    a.sched_nsplit[b] = ns;
    a.sched_base[b] = base;
    for (int k = 0; k < ns; ++k) a.sched_map[base + k] = make_int4(b, k, base, P);
    base += ns;
  }
  // the last thread's running prefix is the total chunk count; CTAs past it
  // get no chunk
  __syncthreads();
  if (tid == 127) red[0] = base;
  __syncthreads();
  for (int c = red[0] + tid; c < C; c += 128) a.sched_map[c] = make_int4(-1, 0, 0, 0);
}

template <int NB>
__global__ void __launch_bounds__(128) qprep_kernel(DecodeArgs a, const float* __restrict__ RK,
                                                    const float* __restrict__ mu,
                                                    float log2_scale) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  griddep_launch_dependents();
  const int b0 = blockIdx.x * NB;
  if (b0 >= a.batch) {               // the extra column of a balanced decode
    if (blockIdx.y == 0)
      schedule_cta(a, reinterpret_cast<int*>(smem_raw), static_cast<int>(sizeof(QprepSmem<NB>) / 4));
    return;
  }
  qprep_cta<NB>(a, RK, mu, log2_scale, *reinterpret_cast<QprepSmem<NB>*>(smem_raw), b0,
                min(NB, a.batch - b0), blockIdx.y);
}

// ---------------------------------------------------------------------------
// Append + query preparation in one launch (kvq_append_decode), CTA (group of
// sequences, kv, role).  Roles 0 and 1 quantise the new key and the new value
// (position seq_lens[b] - 1) of each sequence b of the group for KV head kv
// into its page record, with exactly the fp32 operation sequence of the
// append kernel (centre the key, fmaf chain over j = 0..127 in order,
// max/min, clip, fp16 scale/zero, rint codes); the other roles prepare the
// rotated queries exactly like qprep_kernel.  The roles share nothing, so
// they run side by side.  Rotation matrices are bulk-copied before the CTA
// waits for its predecessor; the token, q and the tables are read, and the
// pool written, only after that wait.
// ---------------------------------------------------------------------------
template <int NB>
struct StepSmem {
  float R[kDim * kDim];              // R_K (key role) or R_V (value role)
  alignas(16) float x[NB][kDim];     // the centred key or the value of each sequence, then its rotation
  float red[NB][2][4];               // [sequence][max|min][warp]
  uint8_t codes[NB][kDim];
  uint8_t* rec[NB];                  // the page record of the sequence's new token, or none
  uint8_t* bf16_rec[NB];             // its BF16 window record, or none
  int tau[NB];                       // the token's row in its page
  uint32_t szw[NB];                  // fp16 scale | fp16 zero << 16
  uint64_t bar;
};

// Sequences per query CTA of a step preparation whose append CTAs take NB:
// the query rotation costs G times the append's per sequence, so its groups
// stay small and more of its CTAs share the wave.
template <int NB>
__host__ __device__ constexpr int step_query_nb() { return NB < 2 ? NB : 2; }
template <int NB>
__host__ __device__ constexpr int step_roles() { return 2 + NB / step_query_nb<NB>(); }

template <int NB>
union StepPrepSmem {
  StepSmem<NB> append;
  QprepSmem<step_query_nb<NB>()> query;
};

// CTA (group of NB sequences, kv, role): role 0 appends the new keys of the
// group's sequences for KV head kv, role 1 their new values, roles 2, 3, ...
// prepare their queries, step_query_nb<NB>() sequences each (every role
// stages its one rotation matrix, so every CTA of the launch needs at most
// one matrix of shared memory and several fit on an SM).
template <int NB>
__global__ void __launch_bounds__(128) step_prep_kernel(DecodeArgs a, StepArgs st) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int b0 = blockIdx.x * NB, kv = blockIdx.y, i = threadIdx.x;
  griddep_launch_dependents();
  if (b0 >= a.batch) {               // the extra column of a balanced decode
    if (kv == 0 && blockIdx.z == 0)
      schedule_cta(a, reinterpret_cast<int*>(smem_raw), static_cast<int>(sizeof(StepPrepSmem<NB>) / 4));
    return;
  }
  const int nb = min(NB, a.batch - b0);
  if (blockIdx.z >= 2) {
    constexpr int NBQ = step_query_nb<NB>();
    const int bq = b0 + (blockIdx.z - 2) * NBQ;
    if (bq < a.batch)
      qprep_cta<NBQ>(a, st.q_rotated ? nullptr : st.RK, st.mu, a.log2_scale,
                     reinterpret_cast<StepPrepSmem<NB>*>(smem_raw)->query, bq,
                     min(NBQ, a.batch - bq), kv);
    return;
  }
  const int which = blockIdx.z;      // 0 keys, 1 values
  StepSmem<NB>& sm = reinterpret_cast<StepPrepSmem<NB>*>(smem_raw)->append;
  const int warp = i >> 5, lane = i & 31;
  const uint32_t bar = smem_u32(&sm.bar);
  if (i == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, kDim * kDim * 4);
    bulk_g2s(smem_u32(sm.R), (which ? st.RV : st.RK) + static_cast<size_t>(kv) * kDim * kDim,
             kDim * kDim * 4, bar);
  }
  __syncthreads();
  griddep_wait();      // tokens and tables may come from preceding kernels

  const float mui = which ? 0.0f : st.mu[static_cast<size_t>(kv) * kDim + i];
  const uint16_t* X = which ? st.V : st.K;
  // element i of each sequence's token, then (lane u of warp 0) the page
  // lookups of sequence u, in the same round trip; per-sequence loops below
  // run from shared memory, so that the kernel's code stays small
  uint16_t bits[NB];
#pragma unroll
  for (int u = 0; u < NB; ++u)
    bits[u] = u < nb ? X[(static_cast<size_t>(b0 + u) * a.Hkv + kv) * kDim + i] : 0;
  if (warp == 0 && lane < NB) {
    const int u = lane;
    uint8_t* rec = nullptr;
    uint8_t* brec = nullptr;
    int tau = 0;
    if (u < nb) {
      const int b = b0 + u;
      const int seq_len = a.seq_lens[b];
      const int p = seq_len - 1;
      if (seq_len > a.max_pages * kPage) {
        if (kv == 0 && which == 0) atomicOr(a.status, KVQ_STATUS_BAD_SEQLEN);
      } else if (p >= 0) {
        tau = p % kPage;
        const int page = a.page_table[static_cast<size_t>(b) * a.max_pages + p / kPage];
        if (page >= 0 && page < a.num_pool_pages)
          rec = st.pool + (static_cast<size_t>(page) * a.Hkv + kv) * kInt2Rec;
        else if (which == 0)
          atomicOr(a.status, KVQ_STATUS_BAD_PAGE);
        if (st.bf16_pool != nullptr) {
          const int bpage = st.bf16_page_table[static_cast<size_t>(b) * a.max_pages + p / kPage];
          if (bpage >= 0 && bpage < st.bf16_num_pool_pages)
            brec = st.bf16_pool + (static_cast<size_t>(bpage) * a.Hkv + kv) * kBf16Rec;
          else if (which == 0)
            atomicOr(a.status, KVQ_STATUS_BAD_PAGE);
        }
      }
    }
    sm.rec[u] = rec;
    sm.bf16_rec[u] = brec;
    sm.tau[u] = tau;
  }
#pragma unroll
  for (int u = 0; u < NB; ++u) {
    const float xf = __uint_as_float(static_cast<uint32_t>(bits[u]) << 16);
    sm.x[u][i] = u < nb ? (which ? xf : __fsub_rn(xf, mui)) : 0.0f;
  }
  __syncthreads();
  // the BF16 window cache's copy of each token (same placement as the BF16
  // append kernel: fragment order of the BF16 page record)
  if (st.bf16_pool != nullptr) {
#pragma unroll 1
    for (int u = 0; u < nb; ++u) {
      uint8_t* base = sm.bf16_rec[u];
      if (base == nullptr) continue;
      const int tau = sm.tau[u];
      const uint16_t bu = X[(static_cast<size_t>(b0 + u) * a.Hkv + kv) * kDim + i];
      if (which == 0) {
        const int w = i >> 4, r = i & 15, h = r >> 3, t = (r >> 1) & 3, e = r & 1;
        const int L = 4 * (tau & 7) + t, reg = (tau >> 3) + 2 * h;
        *reinterpret_cast<uint16_t*>(base + 512 * w + 16 * L + 4 * reg + 2 * e) = bu;
      } else {
        const int m = i >> 4, r = i & 15, g = r & 7, dh = r >> 3;
        const int t = (tau & 7) >> 1, e = tau & 1, th = tau >> 3;
        const int L = 4 * g + t, reg = 2 * th + dh;
        *reinterpret_cast<uint16_t*>(base + 4096 + 512 * m + 16 * L + 4 * reg + 2 * e) = bu;
      }
    }
  }
  const bool ok = mbar_wait_bounded(bar, 0);
  if (__syncthreads_or(!ok)) {
    if (i == 0) {
      atomicOr(a.status, KVQ_STATUS_TIMEOUT);
      mbar_drain(bar, 0);
    }
    return;
  }
  // r_i = fmaf chain over j = 0..127 per sequence, the vector elements read
  // four j at a time; the chains of the group's sequences side by side
  {
    float r[NB];
#pragma unroll
    for (int u = 0; u < NB; ++u) r[u] = 0.0f;
#pragma unroll 2
    for (int j0 = 0; j0 < kDim; j0 += 4) {
      float r4[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) r4[k] = sm.R[(j0 + k) * kDim + i];
#pragma unroll
      for (int u = 0; u < NB; ++u) {
        const float4 x = *reinterpret_cast<const float4*>(&sm.x[u][j0]);
        r[u] = fmaf(x.x, r4[0], r[u]);
        r[u] = fmaf(x.y, r4[1], r[u]);
        r[u] = fmaf(x.z, r4[2], r[u]);
        r[u] = fmaf(x.w, r4[3], r[u]);
      }
    }
    __syncthreads();                 // every thread is done reading the vectors
#pragma unroll
    for (int u = 0; u < NB; ++u) sm.x[u][i] = r[u];
  }
  // max / min of each rotated vector over its 128 elements
#pragma unroll 1
  for (int u = 0; u < nb; ++u) {
    float mx = sm.x[u][i], mn = mx;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    }
    if (lane == 0) {
      sm.red[u][0][warp] = mx;
      sm.red[u][1][warp] = mn;
    }
  }
  __syncthreads();
  const float clip = which ? st.clip_v : st.clip_k;
#pragma unroll 1
  for (int u = 0; u < nb; ++u) {
    const float mx = fmaxf(fmaxf(sm.red[u][0][0], sm.red[u][0][1]),
                           fmaxf(sm.red[u][0][2], sm.red[u][0][3]));
    const float mn = fminf(fminf(sm.red[u][1][0], sm.red[u][1][1]),
                           fminf(sm.red[u][1][2], sm.red[u][1][3]));
    const float mxc = __fmul_rn(clip, mx);
    const float mnc = __fmul_rn(clip, mn);
    const float s32 = __fdiv_rn(__fsub_rn(mxc, mnc), 3.0f);
    const __half sh = __float2half_rn(s32);
    const __half zh = __float2half_rn(mnc);
    const float sc = __half2float(sh), z = __half2float(zh);
    uint32_t code = 0;
    if (sc != 0.0f) {
      const float t = __fdiv_rn(__fsub_rn(sm.x[u][i], z), sc);
      code = static_cast<uint32_t>(fminf(fmaxf(rintf(t), 0.0f), 3.0f));
    }
    sm.codes[u][i] = static_cast<uint8_t>(code);
    if (i == 0)
      sm.szw[u] = static_cast<uint32_t>(__half_as_ushort(sh)) |
                  (static_cast<uint32_t>(__half_as_ushort(zh)) << 16);
  }
  __syncthreads();
  // scatter this role's half of each page record (layout in include/kvq.h)
#pragma unroll 1
  for (int u = 0; u < nb; ++u) {
    uint8_t* const rp = sm.rec[u];
    if (rp == nullptr) continue;
    const int tau = sm.tau[u];
    if (which == 0 && i < 8) {
      // keys: word h of lane group t of row tau & 7
      const int t = i & 3, h = i >> 2;
      uint32_t wv = 0;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const int d = 16 * w + 2 * t + 8 * h;
        wv |= static_cast<uint32_t>(sm.codes[u][d]) << (2 * w);
        wv |= static_cast<uint32_t>(sm.codes[u][d + 1]) << (16 + 2 * w);
      }
      *reinterpret_cast<uint32_t*>(rp + 16 * (4 * (tau & 7) + t) + 8 * (tau >> 3) + 4 * h) = wv;
    } else if (which == 1 && i < 16) {
      // values: the token's 16-bit half of word (2 th + dh) of lane 4 g + t
      const int g = i >> 1, dh = i & 1;
      uint32_t hv = 0;
#pragma unroll
      for (int m = 0; m < 8; ++m) hv |= static_cast<uint32_t>(sm.codes[u][16 * m + g + 8 * dh]) << (2 * m);
      const int t = (tau & 7) >> 1, e = tau & 1, th = tau >> 3;
      *reinterpret_cast<uint16_t*>(rp + 512 + 16 * (4 * g + t) + 4 * (2 * th + dh) + 2 * e) =
          static_cast<uint16_t>(hv);
    } else if (i == 32) {
      *reinterpret_cast<uint32_t*>(rp + 1024 + 16 * (tau & 7) + 8 * which + 4 * (tau >> 3)) =
          sm.szw[u];
    }
  }
}

// ---------------------------------------------------------------------------
// INT2 split-K decode kernel.
// ---------------------------------------------------------------------------

// fp16x2 operand of code position P (0..7) of a fragment word: the fields at
// bits [2P, 2P+1] and [16+2P, 17+2P], each moved to bit offset B of its half
// and isolated by one AND.  A half whose only set bits lie in [0, 10) is the
// fp16 number (bits) * 2^-24 (subnormal, or the smallest normal binade), so
// the field is exactly code * 2^(B - 24).  Tensor cores keep fewer product bits
// the further the field sits below bit 9, about one bit per place (measured on
// GB300: relative error of a 128-term score 3e-7 with fields at offsets 4..8,
// 1e-5 at offset 0; of a 16-token value sum 2.6e-6 at offset 4, 4e-5 at
// offset 0).  Fields 2-4 are used where they are (offsets 4, 6, 8), fields 0-1
// shifted left by 6 and fields 5-7 right by 6: two shifts and eight ANDs per
// word of 16 codes.
template <int P, int B>
__device__ __forceinline__ uint32_t field_op(uint32_t w) {
  static_assert(B >= 0 && B + 1 < 10, "the field stays below the exponent's second bit");
  constexpr uint32_t kM = (3u << B) | (3u << (B + 16));
  constexpr int kShift = B - 2 * P;
  if constexpr (kShift > 0) return (w << kShift) & kM;
  else if constexpr (kShift < 0) return (w >> (-kShift)) & kM;
  else return w & kM;
}
template <int P>
__device__ __forceinline__ uint32_t code_op(uint32_t w) { return field_op<P, code_bit(P)>(w); }

// Scores of one page for this lane: tokens g and g+8 of head t (qc, before the
// per-token scale/zero).  kw: the lane's K-code words {tok g h0, tok g h1,
// tok g+8 h0, tok g+8 h1}; A fragment = {tok g lo dims, tok g+8 lo, tok g hi,
// tok g+8 hi}.
__device__ __forceinline__ void page_scores(const uint4& kw, const uint32_t (&qf)[16],
                                            float (&s)[4]) {
#define KVQ_KSTEP(ACC, P) \
  mma_f16(ACC, code_op<P>(kw.x), code_op<P>(kw.z), code_op<P>(kw.y), code_op<P>(kw.w), \
          qf[2 * (P)], qf[2 * (P) + 1])
  // one accumulator chain per page (the pair's two pages are independent
  // chains; two chains per page cost four adds and four zeroings more)
  s[0] = s[1] = s[2] = s[3] = 0.0f;
  KVQ_KSTEP(s, 0); KVQ_KSTEP(s, 1); KVQ_KSTEP(s, 2); KVQ_KSTEP(s, 3);
  KVQ_KSTEP(s, 4); KVQ_KSTEP(s, 5); KVQ_KSTEP(s, 6); KVQ_KSTEP(s, 7);
#undef KVQ_KSTEP
}

// O^T[dims][cols] += Vcode^T . P for one page.  vw: the lane's V-code words
// {toks 2t|2t+1 dim g, dim g+8, toks 2t+8|2t+9 dim g, dim g+8}.
__device__ __forceinline__ void page_values(const uint4& vw, uint32_t pb0, uint32_t pb1,
                                            float (&acc)[8][4]) {
#define KVQ_VSTEP(P) \
  mma_f16(acc[P], code_op<P>(vw.x), code_op<P>(vw.y), code_op<P>(vw.z), code_op<P>(vw.w), pb0, pb1)
  KVQ_VSTEP(0); KVQ_VSTEP(1); KVQ_VSTEP(2); KVQ_VSTEP(3);
  KVQ_VSTEP(4); KVQ_VSTEP(5); KVQ_VSTEP(6); KVQ_VSTEP(7);
#undef KVQ_VSTEP
}

// P - float(h) for the two halves h of X, each in one mixed-precision fma
// (f16 x f16 + f32: h * -1 + P, the f16 operands widened exactly).
__device__ __forceinline__ void half2_residuals(uint32_t X, float P0, float P1, float& r0,
                                                float& r1) {
  asm("{\n\t.reg .f16 a, b, m;\n\t"
      "mov.b32 {a, b}, %2;\n\t"
      "mov.b16 m, 0xBC00;\n\t"
      "fma.rn.f32.f16 %0, a, m, %3;\n\t"
      "fma.rn.f32.f16 %1, b, m, %4;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "r"(X), "f"(P0), "f"(P1));
}

// B fragments of the value product from this lane's weights of tokens g and
// g+8 (head t): column 2*head holds the fp16 weight X = fp16(P), column
// 2*head+1 the fp16 residual (P - X) * 2^11 (P - X is exact in fp32; the 2^11
// keeps the residual a normal fp16 number down to P = 2^-14, so weights far
// below the running max keep about 22 bits; the epilogue scales that column
// back).  The lane's pairs {weight, residual} of token g (and of token g+8)
// are row g, columns 2t and 2t+1 of an 8 x 8 matrix of 16-bit values (rows =
// tokens, columns = 2*head + part) in mma fragment order; its transpose
// (movmatrix) gives lane (g, t) tokens 2t and 2t+1 of column g, which is the B
// fragment.
__device__ __forceinline__ void weights_to_b(float P0, float P1, uint32_t& pb0, uint32_t& pb1) {
  const uint32_t X = pack_half2(P0, P1);
  float r0, r1;
  half2_residuals(X, P0, P1, r0, r1);
  const uint32_t Y = pack_half2(r0 * 2048.0f, r1 * 2048.0f);
  pb0 = movmatrix_trans(__byte_perm(X, Y, 0x5410));
  pb1 = movmatrix_trans(__byte_perm(X, Y, 0x7632));
}

// Weights are kept <= 2^kLazy relative to the running max before it is raised.
constexpr float kLazy = 8.0f;

// Online-softmax update with one pair of pages (A, B) of a stage for this lane:
// scores, running max, weights, value accumulation.  kMasked = false is the
// common case of two full, valid pages: no per-token masks at all.
struct WarpState {
  float acc[8][4];
  float m_run, l_run, z_run;
  float F;                   // rescale factor owed by the flushed total (see flush_acc)
};

template <bool kMasked>
__device__ __forceinline__ void process_pair(WarpState& st, const uint32_t (&qf)[16], float kappa,
                                             float zeta, int g, int t, const uint4& kwa,
                                             const uint4& vwa, const uint4& mta, const uint4& kwb,
                                             const uint4& vwb, const uint4& mtb, bool va0, bool va1,
                                             bool vb0, bool vb1) {
  if (!kMasked) va0 = va1 = vb0 = vb1 = true;
  float (&acc)[8][4] = st.acc;
  float& m_run = st.m_run;
  float& l_run = st.l_run;
  float& z_run = st.z_run;
    // ---- scores of both pages (independent tensor-core chains)
    float sa4[4], sb4[4];
    page_scores(kwa, qf, sa4);
    page_scores(kwb, qf, sb4);
    // logit (log2 units) = kappa * s_k * qc + zeta * z_k; qc = hi col + 2^-11 lo col
    const float la0 = va0 ? fmaf(kappa * half_lo(mta.x), fmaf(sa4[1], 1.0f / 2048.0f, sa4[0]),
                                 zeta * half_hi(mta.x)) : -INFINITY;
    const float la1 = va1 ? fmaf(kappa * half_lo(mta.y), fmaf(sa4[3], 1.0f / 2048.0f, sa4[2]),
                                 zeta * half_hi(mta.y)) : -INFINITY;
    const float lb0 = vb0 ? fmaf(kappa * half_lo(mtb.x), fmaf(sb4[1], 1.0f / 2048.0f, sb4[0]),
                                 zeta * half_hi(mtb.x)) : -INFINITY;
    const float lb1 = vb1 ? fmaf(kappa * half_lo(mtb.y), fmaf(sb4[3], 1.0f / 2048.0f, sb4[2]),
                                 zeta * half_hi(mtb.y)) : -INFINITY;

    // ---- online softmax.  The value weights P = p * s_v feed fp16 operands, so
    // the running max m is kept over lv = logit + log2(max(s_v, 2^-24)) and
    // raised only when some lv exceeds m + kLazy: then p * s_v <= 2^kLazy for
    // every token seen.  m_run holds m - 6, so p = 2^(logit - m_run) already
    // carries the weight scale 2^(14 - kLazy) = 2^6 and P = p * max(s_v, 2^-24)
    // stays below 2^14 (max() changes nothing: fp16 s_v is 0 or >= 2^-24, and
    // s_v = 0 gives code 0).  p itself may be large (at most 2^(kLazy + 30)); it
    // is only summed in fp32, and l_run, z_run carry the 2^6 too (removed in
    // the epilogue).  The test lv > m + kLazy is taken as P > 2^14 on the
    // weights against the current max (true for p = inf while m is -inf), so
    // the logarithms are computed only on the rare stages that raise m.
    static_assert(kLazy == 8.0f, "P <= 2^14 is p * s_v <= 2^kLazy with the 2^6 scale");
    const float sva0 = half_lo(mta.z), sva1 = half_lo(mta.w);
    const float svb0 = half_lo(mtb.z), svb1 = half_lo(mtb.w);
    constexpr float kSvMin = 0x1p-24f;
    const float sa0 = fmaxf(sva0, kSvMin), sa1 = fmaxf(sva1, kSvMin);
    const float sb0 = fmaxf(svb0, kSvMin), sb1 = fmaxf(svb1, kSvMin);
    float pa0 = va0 ? fast_exp2(la0 - m_run) : 0.0f;
    float pa1 = va1 ? fast_exp2(la1 - m_run) : 0.0f;
    float pb0v = vb0 ? fast_exp2(lb0 - m_run) : 0.0f;
    float pb1v = vb1 ? fast_exp2(lb1 - m_run) : 0.0f;
    float Pa0 = va0 ? pa0 * sa0 : 0.0f, Pa1 = va1 ? pa1 * sa1 : 0.0f;
    float Pb0 = vb0 ? pb0v * sb0 : 0.0f, Pb1 = vb1 ? pb1v * sb1 : 0.0f;
    const float cmax = fmaxf(fmaxf(Pa0, Pa1), fmaxf(Pb0, Pb1));
    if (__any_sync(0xffffffffu, !(cmax <= 0x1p14f))) {
      const float lva0 = la0 + fmaxf(fast_log2(sva0), -24.0f);
      const float lva1 = la1 + fmaxf(fast_log2(sva1), -24.0f);
      const float lvb0 = lb0 + fmaxf(fast_log2(svb0), -24.0f);
      const float lvb1 = lb1 + fmaxf(fast_log2(svb1), -24.0f);
      const float lmax = fmaxf(fmaxf(lva0, lva1), fmaxf(lvb0, lvb1));
      float pm = lmax;
      pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 4));
      pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 8));
      pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));
      const float pms = pm - 6.0f;
      if (pms > m_run) {
        const float f = fast_exp2(m_run - pms);
#pragma unroll
        for (int mb = 0; mb < 8; ++mb)
#pragma unroll
          for (int q = 0; q < 4; ++q) acc[mb][q] *= f;
        l_run *= f;
        z_run *= f;
        st.F *= f;
        m_run = pms;
      }
      pa0 = va0 ? fast_exp2(la0 - m_run) : 0.0f;
      pa1 = va1 ? fast_exp2(la1 - m_run) : 0.0f;
      pb0v = vb0 ? fast_exp2(lb0 - m_run) : 0.0f;
      pb1v = vb1 ? fast_exp2(lb1 - m_run) : 0.0f;
      Pa0 = va0 ? pa0 * sa0 : 0.0f;
      Pa1 = va1 ? pa1 * sa1 : 0.0f;
      Pb0 = vb0 ? pb0v * sb0 : 0.0f;
      Pb1 = vb1 ? pb1v * sb1 : 0.0f;
    }
    l_run += (pa0 + pa1) + (pb0v + pb1v);
    if (va0) z_run = fmaf(pa0, half_hi(mta.z), z_run);
    if (va1) z_run = fmaf(pa1, half_hi(mta.w), z_run);
    if (vb0) z_run = fmaf(pb0v, half_hi(mtb.z), z_run);
    if (vb1) z_run = fmaf(pb1v, half_hi(mtb.w), z_run);

    // ---- values of both pages
    uint32_t fa0, fa1, fb0, fb1;
    weights_to_b(Pa0, Pa1, fa0, fa1);
    weights_to_b(Pb0, Pb1, fb0, fb1);
    page_values(vwa, fa0, fa1, acc);
    page_values(vwb, fb0, fb1, acc);
}

constexpr int kW = kInt2Warps;                 // warps per CTA
constexpr int kPPS = 4;                        // pages per stage (two pairs)
constexpr int kNS = 2;                         // pipeline stages per warp
constexpr int kMaxIds = 1024;                  // page ids staged per sub-chunk
constexpr int kFlushStages = 16;               // stages between accumulator flushes

// The tensor cores' fp32 accumulation of P.V is not round-to-nearest: over many
// pages the running accumulator drifts (about 2e-4 relative after 1,300 pages
// of one split).  Every kFlushStages stages each lane adds its accumulator
// into its own fp32 total in shared memory (round-to-nearest fma) and restarts
// it from zero; F carries the running-max rescales made since the last flush.
__device__ __forceinline__ void flush_acc(WarpState& ws, float* tot) {
#pragma unroll
  for (int mb = 0; mb < 8; ++mb)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float* p = tot + 32 * (4 * mb + q);
      *p = fmaf(*p, ws.F, ws.acc[mb][q]);
      ws.acc[mb][q] = 0.0f;
    }
  ws.F = 1.0f;
}

// Every warp streams its own KV head's records through its own ring: no stage
// is shared between warps, so no warp waits for another to release a slot.
struct Int2Merge {
  float o[kW][kMaxG][kDim];
  float m[kW][kMaxG];
  float l[kW][kMaxG];
};
struct Int2Smem {
  union {
    uint8_t ring[kW][kNS][kPPS * kInt2Rec];
    Int2Merge mg;
  };
  uint64_t full[kW][kNS];
  int ids[kMaxIds];
  float tot[kW][32][32];     // per warp and lane: flushed P.V totals, [acc index][lane]
};

// Fill stage k of warp `warp`: pages kPPS*k .. kPPS*k + kPPS - 1 of the warp's
// share of the sub-chunk, one bulk copy per page.  idw: the warp's page ids,
// contiguous and 16-byte aligned (one shared load per stage); a record is at
// pool_kv + id * stride.  Lane 0 only.
__device__ __forceinline__ void issue_warp_stage(Int2Smem& sm, const int* idw, int warp, int k,
                                                  int slot, int npw, const uint8_t* pool_kv,
                                                  uint32_t stride) {
  const int4 v = *reinterpret_cast<const int4*>(idw + kPPS * k);
  const uint32_t bar = smem_u32(&sm.full[warp][slot]);
  const uint32_t dst = smem_u32(&sm.ring[warp][slot][0]);
  int id[kPPS] = {v.x, v.y, v.z, v.w};
  uint32_t bytes = 0;
#pragma unroll
  for (int u = 0; u < kPPS; ++u) {
    if (kPPS * k + u >= npw) id[u] = -1;
    bytes += id[u] >= 0 ? kInt2Rec : 0;
  }
  if (bytes == 0) {
    mbar_arrive(bar);
    return;
  }
  mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
  for (int u = 0; u < kPPS; ++u)
    if (id[u] >= 0)
      bulk_g2s(dst + u * kInt2Rec,
               pool_kv + static_cast<uint64_t>(static_cast<uint32_t>(id[u])) * stride, kInt2Rec, bar);
}

// kBalanced: CTA (c, hg) takes the chunk that the balanced schedule assigns to
// c (DecodeArgs::sched_map); otherwise CTA (split, hg, b) takes chunk `split`
// of sequence b, chunk_pages pages each.
template <bool kBalanced>
__global__ void __launch_bounds__(kW * 32, 2) decode_int2_kernel(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Int2Smem& sm = *reinterpret_cast<Int2Smem*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  const int hg = blockIdx.y;
  const int HPC = a.hpc, GPH = kW / HPC;
  const int hl = warp / GPH, gi = warp % GPH;
  const int kv = hg * HPC + hl;

  if (lane == 0) {
    for (int s = 0; s < kNS; ++s) mbar_init(smem_u32(&sm.full[warp][s]), 1);
    fence_mbar_init();
  }
  griddep_wait();      // inputs (pool, tables, rotated queries) come from predecessors
  int split, b, chunk_pages, slot0;
  if constexpr (kBalanced) {
    const int4 m = a.sched_map[blockIdx.x];
    if (m.x < 0) return;             // no chunk for this CTA (nothing issued yet)
    b = m.x;
    split = m.y;
    slot0 = m.z;
    chunk_pages = m.w;
  } else {
    split = blockIdx.x;
    b = blockIdx.z;
    slot0 = 0;
    chunk_pages = a.chunk_pages;
  }
  // split partial of head `head` (of sequence b)
  auto part_of = [&](int head) -> float* {
    return kBalanced ? a.part + (static_cast<size_t>(slot0 + split) * a.H + head) * kPartStride
                     : a.part + ((static_cast<size_t>(b) * a.H + head) * a.splits + split) * kPartStride;
  };

  // INT2 tokens: positions [lo, hi); with a BF16 window the first win_sink and
  // the last win_recent positions are left to the window pass.
  const int lo = a.win_sink;
  const int p0 = max(split * chunk_pages, lo / kPage);
  const int32_t* ptab = a.page_table + static_cast<size_t>(b) * a.max_pages;
  // The first sub-chunk's page ids are loaded together with seq_len (one round
  // trip instead of two): every entry of the split's chunk inside the table,
  // of which those below the sequence's end are used.
  constexpr int kIdsPerThread = kMaxIds / (kW * 32);
  const int nspec = min(kMaxIds, max(0, min(split * chunk_pages + chunk_pages, a.max_pages) - p0));
  int spec[kIdsPerThread];
#pragma unroll
  for (int r = 0; r < kIdsPerThread; ++r) {
    const int i = tid + r * kW * 32;
    spec[r] = i < nspec ? ptab[p0 + i] : -1;
  }
  int seq_len = a.seq_lens[b];
  if (seq_len < 0 || seq_len > a.max_pages * kPage) {
    if (tid == 0 && split == 0 && hg == 0) atomicOr(a.status, KVQ_STATUS_BAD_SEQLEN);
    seq_len = 0;
  }
  const int hi = max(seq_len - a.win_recent, 0);
  const int n_pages = (hi + kPage - 1) / kPage;      // <= max_pages, so npg <= nspec
  const int npg = max(0, min(split * chunk_pages + chunk_pages, n_pages) - p0);

  // B fragments of the rotated query and the head's logit constants
  uint32_t qf[16];
  {
    const uint4* src = reinterpret_cast<const uint4*>(
        a.qfrag + ((static_cast<size_t>(b) * a.Hkv + kv) * 32 + lane) * 16);
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const uint4 v = src[r];
      qf[4 * r] = v.x; qf[4 * r + 1] = v.y; qf[4 * r + 2] = v.z; qf[4 * r + 3] = v.w;
    }
  }
  const float kappa = a.qmeta[(static_cast<size_t>(b) * a.Hkv + kv) * kQMeta + 2 * t];
  const float zeta = a.qmeta[(static_cast<size_t>(b) * a.Hkv + kv) * kQMeta + 2 * t + 1];

  WarpState ws;
#pragma unroll
  for (int mb = 0; mb < 8; ++mb)
#pragma unroll
    for (int k = 0; k < 4; ++k) ws.acc[mb][k] = 0.0f;
  ws.m_run = -INFINITY;
  ws.l_run = 0.0f;
  ws.z_run = 0.0f;

  ws.F = 1.0f;
  float* const tot = &sm.tot[warp][0][lane];
#pragma unroll
  for (int j = 0; j < 32; ++j) tot[32 * j] = 0.0f;

  const uint8_t* const pool_kv = a.pool + static_cast<size_t>(kv) * kInt2Rec;
  const uint32_t rec_stride = static_cast<uint32_t>(a.Hkv) * kInt2Rec;   // <= 64 x 1152
  int gs = 0;            // this warp's stages consumed so far (ring phase)
  bool timed_out = false;
  // after a wait gave up: this warp's stages still in flight, [drain_k, drain_end)
  // of the sub-chunk whose stages start at ring position drain_base
  int drain_k = 0, drain_end = 0, drain_base = 0;
  for (int sub = 0; sub < npg && !timed_out; sub += kMaxIds) {
    const int nsub = min(kMaxIds, npg - sub);
    bool ids_ok = true;
#pragma unroll
    for (int r = 0; r < kIdsPerThread; ++r) {
      const int i = tid + r * kW * 32;
      if (i < nsub) {
        const int id = sub == 0 ? spec[r] : ptab[p0 + sub + i];
        const bool ok = id >= 0 && id < a.num_pool_pages;
        if (!ok) atomicOr(a.status, KVQ_STATUS_BAD_PAGE);
        // local page i goes to warp i % GPH of its head as that warp's page
        // i / GPH: each warp's ids are contiguous
        sm.ids[(i & (GPH - 1)) * (kMaxIds / GPH) + i / GPH] = ok ? id : -1;
        ids_ok = ids_ok && ok;
      }
    }
    const bool all_ids_ok = __syncthreads_and(ids_ok);
    const int npw = nsub > gi ? (nsub - gi + GPH - 1) / GPH : 0;   // this warp's pages
    const int nst = (npw + kPPS - 1) / kPPS;
    const int* idw = sm.ids + gi * (kMaxIds / GPH);
    // pairs (j, j + 1) with both pages present, valid and all their tokens in
    // [lo, hi): jlo <= j < jend (page of warp page j: c + GPH j)
    int jlo = 0, jend = 0;
    {
      const int c = p0 + sub + gi;
      const int L = (lo + kPage - 1) / kPage;
      jlo = L > c ? (L - c + GPH - 1) / GPH : 0;
      const int tt = hi / kPage - 1 - c;
      jend = (all_ids_ok && tt >= 0) ? min(npw - 1, tt / GPH) : 0;
    }
    if (lane == 0)
      for (int k = 0; k < kNS && k < nst; ++k)
        issue_warp_stage(sm, idw, warp, k, (gs + k) % kNS, npw, pool_kv, rec_stride);

    for (int k = 0; k < nst; ++k) {
      const int slot = (gs + k) % kNS;
      if (!mbar_wait_bounded(smem_u32(&sm.full[warp][slot]), ((gs + k) / kNS) & 1)) {
        if (lane == 0) atomicOr(a.status, KVQ_STATUS_TIMEOUT);
        timed_out = true;
        // stages k .. k + kNS - 1 (those below nst) have been issued
        drain_k = k;
        drain_end = min(k + kNS, nst);
        drain_base = gs;
        break;
      }
      static_assert(kPPS % 2 == 0, "stages hold whole pairs of pages");
#pragma unroll
      for (int h = 0; h < kPPS / 2; ++h) {
        const int j = kPPS * k + 2 * h;            // the warp's page index of page a
        const int ua = gi + GPH * j, ub = ua + GPH;
        const uint8_t* sta = &sm.ring[warp][slot][2 * h * kInt2Rec];
        const uint8_t* stb = sta + kInt2Rec;
        const uint4 kwa = *reinterpret_cast<const uint4*>(sta + 16 * lane);
        const uint4 vwa = *reinterpret_cast<const uint4*>(sta + 512 + 16 * lane);
        const uint4 mta = *reinterpret_cast<const uint4*>(sta + 1024 + 16 * g);
        const uint4 kwb = *reinterpret_cast<const uint4*>(stb + 16 * lane);
        const uint4 vwb = *reinterpret_cast<const uint4*>(stb + 512 + 16 * lane);
        const uint4 mtb = *reinterpret_cast<const uint4*>(stb + 1024 + 16 * g);
        if (h == kPPS / 2 - 1) {
          __syncwarp();
          if (lane == 0 && k + kNS < nst) {
            fence_proxy_async();
            issue_warp_stage(sm, idw, warp, k + kNS, slot, npw, pool_kv, rec_stride);
          }
        }
        if (j >= npw) continue;
        // both pages present, valid and all their tokens in [lo, hi)
        const bool full = j >= jlo && j < jend;
        if (full) {
          process_pair<false>(ws, qf, kappa, zeta, g, t, kwa, vwa, mta, kwb, vwb, mtb, true, true,
                              true, true);
        } else {
          const bool oka = idw[j] >= 0;
          const bool okb = j + 1 < npw && idw[j + 1] >= 0;
          const int posa = (p0 + sub + ua) * kPage, posb = (p0 + sub + ub) * kPage;
          const bool va0 = oka && posa + g >= lo && posa + g < hi;
          const bool va1 = oka && posa + g + 8 >= lo && posa + g + 8 < hi;
          const bool vb0 = okb && posb + g >= lo && posb + g < hi;
          const bool vb1 = okb && posb + g + 8 >= lo && posb + g + 8 < hi;
          process_pair<true>(ws, qf, kappa, zeta, g, t, kwa, vwa, mta, kwb, vwb, mtb, va0, va1,
                             vb0, vb1);
        }
      }
      if (((gs + k) % kFlushStages) == kFlushStages - 1) flush_acc(ws, tot);
    }
    gs += nst;
    // sm.ids is reloaded for the next sub-chunk; every warp leaves together
    timed_out = __syncthreads_or(timed_out);
  }
  // A wait gave up: let this warp's copies still in flight land (bounded), each
  // on the phase it completes, before the CTA can exit, so no bulk copy targets
  // freed shared memory.
  for (int s = drain_k; s < drain_end; ++s) {
    const int q = drain_base + s;
    mbar_drain(smem_u32(&sm.full[warp][q % kNS]), (q / kNS) & 1);
  }
  griddep_launch_dependents();
  // the flushed totals back into the accumulator
#pragma unroll
  for (int mb = 0; mb < 8; ++mb)
#pragma unroll
    for (int q = 0; q < 4; ++q) ws.acc[mb][q] = fmaf(tot[32 * (4 * mb + q)], ws.F, ws.acc[mb][q]);

  // ---- warp epilogue: (m, l, o) of the warp's KV head for its G query heads
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    ws.l_run += __shfl_xor_sync(0xffffffffu, ws.l_run, off);
    ws.z_run += __shfl_xor_sync(0xffffffffu, ws.z_run, off);
  }
  // undo the code scale 2^(code_bit(mb) - 24) of m-block mb and the weight
  // scale 2^(14 - kLazy) = 2^6 (also on l_run, z_run and m_run); the residual
  // column carries 2^11 more
  static_assert(kLazy == 8.0f, "the value factors below carry the weight scale 2^6");
  if (GPH == 1) {
    // One warp per KV head: its (m, l, o) is the split partial as it stands,
    // stored straight from registers (a merge through shared memory would be a
    // chain of dependent loads on one warp per scheduler).  Same values as the
    // merge below with a single term: an empty head gives (-inf, 0, 0), and
    // "+ 0" turns a -0 into the +0 that merge's fmaf(1, o, 0) gives.
    if (t < a.G) {
      float* p = part_of(kv * a.G + t);
      const bool any = ws.m_run > -INFINITY;
      const float zr = ws.z_run * 0x1p-6f;
#pragma unroll
      for (int mb = 0; mb < 8; ++mb) {
        const float inv = static_cast<float>(1u << (18 - code_bit(mb)));
        const float o0 = fmaf(fmaf(ws.acc[mb][1], 0x1p-11f, ws.acc[mb][0]), inv, zr);
        const float o1 = fmaf(fmaf(ws.acc[mb][3], 0x1p-11f, ws.acc[mb][2]), inv, zr);
        p[4 + 16 * mb + g] = any ? o0 + 0.0f : 0.0f;
        p[4 + 16 * mb + g + 8] = any ? o1 + 0.0f : 0.0f;
      }
      if (g == 0) {
        p[0] = ws.m_run + 6.0f;
        p[1] = any ? ws.l_run * 0x1p-6f : 0.0f;
      }
    }
    return;
  }
  if (t < a.G) {
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) {
      const float inv = static_cast<float>(1u << (18 - code_bit(mb)));
      sm.mg.o[warp][t][16 * mb + g] =
          fmaf(fmaf(ws.acc[mb][1], 0x1p-11f, ws.acc[mb][0]), inv, ws.z_run * 0x1p-6f);
      sm.mg.o[warp][t][16 * mb + g + 8] =
          fmaf(fmaf(ws.acc[mb][3], 0x1p-11f, ws.acc[mb][2]), inv, ws.z_run * 0x1p-6f);
    }
    if (g == 0) {
      sm.mg.m[warp][t] = ws.m_run + 6.0f;
      sm.mg.l[warp][t] = ws.l_run * 0x1p-6f;
    }
  }
  __syncthreads();
  // ---- merge the 8/HPC warps of each head and write the split partials
  for (int idx = tid; idx < HPC * kDim; idx += kW * 32) {
    const int h2 = idx / kDim, d = idx % kDim;
    for (int h = 0; h < a.G; ++h) {
      float M = -INFINITY;
      for (int u = 0; u < GPH; ++u) M = fmaxf(M, sm.mg.m[h2 * GPH + u][h]);
      float L = 0.0f, o = 0.0f;
      if (M > -INFINITY) {
        for (int u = 0; u < GPH; ++u) {
          const int w = h2 * GPH + u;
          if (sm.mg.m[w][h] == -INFINITY) continue;
          const float f = fast_exp2(sm.mg.m[w][h] - M);
          L = fmaf(f, sm.mg.l[w][h], L);
          o = fmaf(f, sm.mg.o[w][h][d], o);
        }
      }
      float* p = part_of((hg * HPC + h2) * a.G + h);
      p[4 + d] = o;
      if (d == 0) {
        p[0] = M;
        p[1] = L;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// BF16 split-K decode kernel (comparison point): per-warp rings of whole
// pages, bf16 operands read straight from the staged page, plain logits
// q.k * sm_scale.  The 4 warps of a CTA take every 4th page of the split.
// ---------------------------------------------------------------------------
struct CtaCombineSmem {
  float o[kDecodeWarps][kMaxG][kDim];
  float m[kDecodeWarps][kMaxG];
  float l[kDecodeWarps][kMaxG];
};

__device__ __forceinline__ void write_partial_bf16(CtaCombineSmem& cs, const DecodeArgs& a, int b,
                                                   int kv, int split) {
  __syncthreads();
  const int d = threadIdx.x;
  for (int h = 0; h < a.G; ++h) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kDecodeWarps; ++w) M = fmaxf(M, cs.m[w][h]);
    float L = 0.0f, o = 0.0f;
    if (M > -INFINITY) {
#pragma unroll
      for (int w = 0; w < kDecodeWarps; ++w) {
        if (cs.m[w][h] == -INFINITY) continue;
        const float f = fast_exp2(cs.m[w][h] - M);
        L = fmaf(f, cs.l[w][h], L);
        o = fmaf(f, cs.o[w][h][d], o);
      }
    }
    float* p = a.part + ((static_cast<size_t>(b) * a.H + kv * a.G + h) * a.splits + split) * kPartStride;
    p[4 + d] = o;
    if (d == 0) {
      p[0] = M;
      p[1] = L;
    }
  }
}

// B fragments of the plain query for the BF16 score product: column g =
// 2*head + part; part 0 carries q (bf16, exact), part 1 is 0.
__device__ __forceinline__ void bf16_q_frags(const DecodeArgs& a, int b, int kv, int g, int t,
                                             uint32_t (&qf)[16]) {
  const int head = g >> 1;
  const bool use = ((g & 1) == 0) && head < a.G;
  const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
      a.q + (static_cast<size_t>(b) * a.H + kv * a.G + (head < a.G ? head : 0)) * kDim);
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    qf[2 * w] = use ? qrow[(16 * w + 2 * t) >> 1] : 0u;
    qf[2 * w + 1] = use ? qrow[(16 * w + 2 * t + 8) >> 1] : 0u;
  }
}

// Online-softmax update of one BF16 page for this lane: s = raw scores of
// tokens g, g+8 (columns 2t, 2t+1 / rows g, g+8 of the C fragment), vf = the
// lane's value A fragments, v0 / v1 = token masks.  The weights enter the value
// product as a bf16 part plus a bf16 residual (columns 2*head, 2*head+1), so
// acc[.][0] + acc[.][1] is the fp32-accurate P.V.
__device__ __forceinline__ void bf16_page_update(const float (&s)[4], const uint4 (&vf)[8],
                                                 bool v0, bool v1, float kappa, int g, int t,
                                                 float (&acc)[8][4], float& m_run, float& l_run) {
  const float l0 = v0 ? kappa * (s[0] + s[1]) : -INFINITY;
  const float l1 = v1 ? kappa * (s[2] + s[3]) : -INFINITY;
  float pm = fmaxf(l0, l1);
  pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 4));
  pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 8));
  pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));
  if (pm > m_run) {
    const float f = fast_exp2(m_run - pm);
#pragma unroll
    for (int mb = 0; mb < 8; ++mb)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc[mb][k] *= f;
    l_run *= f;
    m_run = pm;
  }
  const float P0 = v0 ? fast_exp2(l0 - m_run) : 0.0f;
  const float P1 = v1 ? fast_exp2(l1 - m_run) : 0.0f;
  l_run += P0 + P1;
  const uint32_t X = pack_bf162(P0, P1);
  const float x0 = __uint_as_float(X << 16), x1 = __uint_as_float(X & 0xffff0000u);
  const uint32_t Y = pack_bf162(P0 - x0, P1 - x1);
  const int src0 = 4 * (2 * t) + (g >> 1);
  const uint32_t xa = __shfl_sync(0xffffffffu, X, src0);
  const uint32_t ya = __shfl_sync(0xffffffffu, Y, src0);
  const uint32_t xb = __shfl_sync(0xffffffffu, X, src0 + 4);
  const uint32_t yb = __shfl_sync(0xffffffffu, Y, src0 + 4);
  const uint32_t va = (g & 1) ? ya : xa;
  const uint32_t vb = (g & 1) ? yb : xb;
  const uint32_t pb0 = __byte_perm(va, vb, 0x5410);
  const uint32_t pb1 = __byte_perm(va, vb, 0x7632);
#pragma unroll
  for (int mb = 0; mb < 8; ++mb)
    mma_bf16(acc[mb], vf[mb].x, vf[mb].y, vf[mb].z, vf[mb].w, pb0, pb1);
}

// Per-warp page-id supply: lane j holds the page id of the warp's page 32*blk + j.
struct PageIds {
  int cur, nxt, blk;
};

__device__ __forceinline__ int load_page_id(const int32_t* ptab, int p0, int warp, int count,
                                            int blk, int lane) {
  const int i = 32 * blk + lane;
  return (i < count) ? ptab[p0 + warp + kDecodeWarps * i] : -1;
}

struct Bf16Smem {
  uint8_t ring[kDecodeWarps][kStagesBf16][kBf16Rec];
  uint64_t bar[kDecodeWarps][kStagesBf16];
  int ids[kDecodeWarps][kStagesBf16];
  CtaCombineSmem comb;
};

__global__ void __launch_bounds__(kDecodeThreads, 2) decode_bf16_kernel(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  Bf16Smem& sm = *reinterpret_cast<Bf16Smem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int split = blockIdx.x, kv = blockIdx.y, b = blockIdx.z;

  griddep_wait();
  int seq_len = a.seq_lens[b];
  if (seq_len < 0 || seq_len > a.max_pages * kPage) {
    if (threadIdx.x == 0 && split == 0 && kv == 0) atomicOr(a.status, KVQ_STATUS_BAD_SEQLEN);
    seq_len = 0;
  }
  const int n_pages = (seq_len + kPage - 1) / kPage;
  const int p0 = split * a.chunk_pages;
  const int p1 = min(p0 + a.chunk_pages, n_pages);
  const int count = (p1 - p0 > warp) ? (p1 - p0 - warp + kDecodeWarps - 1) / kDecodeWarps : 0;
  const int32_t* ptab = a.page_table + static_cast<size_t>(b) * a.max_pages;
  const uint8_t* pool_kv = a.pool + static_cast<size_t>(kv) * kBf16Rec;
  const size_t page_stride = static_cast<size_t>(a.Hkv) * kBf16Rec;

  if (lane == 0) {
    for (int s = 0; s < kStagesBf16; ++s) mbar_init(smem_u32(&sm.bar[warp][s]), 1);
    fence_mbar_init();
  }
  __syncwarp();

  PageIds ids;
  ids.blk = 0;
  ids.cur = load_page_id(ptab, p0, warp, count, 0, lane);
  ids.nxt = load_page_id(ptab, p0, warp, count, 1, lane);
  auto issue = [&](int j) {
    if ((j >> 5) != ids.blk) {
      ids.blk = j >> 5;
      ids.cur = ids.nxt;
      ids.nxt = load_page_id(ptab, p0, warp, count, ids.blk + 1, lane);
    }
    const int id = __shfl_sync(0xffffffffu, ids.cur, j & 31);
    if (lane == 0) {
      const int slot = j % kStagesBf16;
      const uint32_t bar = smem_u32(&sm.bar[warp][slot]);
      const bool ok = id >= 0 && id < a.num_pool_pages;
      sm.ids[warp][slot] = ok ? id : -1;
      if (ok) {
        mbar_arrive_expect_tx(bar, kBf16Rec);
        bulk_g2s(smem_u32(sm.ring[warp][slot]), pool_kv + static_cast<size_t>(id) * page_stride,
                 kBf16Rec, bar);
      } else {
        atomicOr(a.status, KVQ_STATUS_BAD_PAGE);
        mbar_arrive(bar);
      }
    }
  };
  for (int j = 0; j < kStagesBf16 && j < count; ++j) issue(j);
  __syncwarp();

  uint32_t qf[16];
  bf16_q_frags(a, b, kv, g, t, qf);
  const float kappa = a.log2_scale;

  float acc[8][4];
#pragma unroll
  for (int mb = 0; mb < 8; ++mb)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[mb][k] = 0.0f;
  float m_run = -INFINITY, l_run = 0.0f;

  int i = 0;
  for (; i < count; ++i) {
    const int slot = i % kStagesBf16;
    const uint32_t parity = (i / kStagesBf16) & 1;
    if (!mbar_wait_bounded(smem_u32(&sm.bar[warp][slot]), parity)) {
      if (lane == 0) atomicOr(a.status, KVQ_STATUS_TIMEOUT);
      break;
    }
    const bool page_ok = sm.ids[warp][slot] >= 0;
    const uint8_t* st = sm.ring[warp][slot];
    const int pos0 = (p0 + warp + kDecodeWarps * i) * kPage;
    const bool v0 = page_ok && (pos0 + g < seq_len);
    const bool v1 = page_ok && (pos0 + g + 8 < seq_len);

    float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const uint4 kf = *reinterpret_cast<const uint4*>(st + 512 * w + 16 * lane);
      mma_bf16(s, kf.x, kf.y, kf.z, kf.w, qf[2 * w], qf[2 * w + 1]);
    }
    uint4 vf[8];
#pragma unroll
    for (int mb = 0; mb < 8; ++mb)
      vf[mb] = *reinterpret_cast<const uint4*>(st + 4096 + 512 * mb + 16 * lane);
    __syncwarp();
    if (i + kStagesBf16 < count) {
      if (lane == 0) fence_proxy_async();
      issue(i + kStagesBf16);
    }
    bf16_page_update(s, vf, v0, v1, kappa, g, t, acc, m_run, l_run);
  }
  if (i < count) {
    // stage i gave up; it and the stages issued after it may still be in flight
    for (int j = i; j < count && j < i + kStagesBf16; ++j)
      mbar_drain(smem_u32(&sm.bar[warp][j % kStagesBf16]), (j / kStagesBf16) & 1);
  }
  griddep_launch_dependents();
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) l_run += __shfl_xor_sync(0xffffffffu, l_run, off);
  if (t < a.G) {
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) {
      sm.comb.o[warp][t][16 * mb + g] = acc[mb][0] + acc[mb][1];
      sm.comb.o[warp][t][16 * mb + g + 8] = acc[mb][2] + acc[mb][3];
    }
    if (g == 0) {
      sm.comb.m[warp][t] = m_run;
      sm.comb.l[warp][t] = l_run;
    }
  }
  write_partial_bf16(sm.comb, a, b, kv, split);
}

// ---------------------------------------------------------------------------
// Log-sum-exp combine of the split partials of the G query heads of one
// (sequence, KV head), then out = o_rot R_V^T.  R_V^T (static data) is staged
// in shared memory by a bulk copy issued before the kernel waits for the decode
// kernel, so the copy overlaps the decode tail.  Warp h reduces the split
// maxima and weights of head h; thread (h, d) then forms element d of head h.
//
// With a BF16 window (kWindow) the kernel first attends, with the plain query,
// over the window tokens of the BF16 cache (the first win_sink and the last
// win_recent positions), before it waits for the decode kernel: those reads
// need nothing from it, and every kernel before it has finished by the time
// the decode kernel lets it launch.  The merge then adds q.mu back to the INT2
// partials (their logits were taken against centred keys) and sums both parts
// in one softmax, in the plain basis (INT2 part rotated back) or, for
// KVQ_OUT_ROTATED, in the rotated one (window part rotated forward by R_V).
// ---------------------------------------------------------------------------
constexpr int kCombineThreads = kMaxG * kDim;   // 512
constexpr int kCombineWarps = kCombineThreads / 32;
static_assert(kCombineThreads == 4 * kDim, "the basis change splits j into four quarters");

struct CombineSmem {
  float Rt[kDim * kDim];      // R_V^T, or R_V for a rotated-basis output with a window
  float w[kMaxG][kMaxSplits];
  alignas(16) float ot[kDim][kMaxG];   // the G outputs, element-major
  float red[4][kMaxG][kDim];           // per-quarter sums of the basis change
  float linv[kMaxG];
  float ww[kMaxG];            // weight of the window part
  uint64_t bar;
};

struct WindowSmem {
  float o[kCombineWarps][kMaxG][kDim];
  float m[kCombineWarps][kMaxG];
  float l[kCombineWarps][kMaxG];
  float M[kMaxG], L[kMaxG];
};

struct CombineWindowSmem {    // dynamic shared memory of combine_kernel<true>
  CombineSmem c;
  WindowSmem win;
};

// BF16 window part of (b, kv): tokens p < win_sink or p >= len - win_recent.
// Warp w takes window pages w, w + 16, ...; each lane loads its fragments of a
// page straight from global memory (the record is in fragment order).  Leaves
// the window maximum / sum per head in ws.M / ws.L and returns, for thread
// (h, d), element d of head h's window output relative to ws.M[h].
__device__ float window_partial(const DecodeArgs& a, WindowSmem& ws, int b, int kv) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;
  int len = a.seq_lens[b];
  if (len < 0 || len > a.max_pages * kPage) len = 0;   // flagged by the decode kernel
  const int sink = min(a.win_sink, len);
  const int rstart = max(len - a.win_recent, 0);       // first recent position
  const int n_pages = (len + kPage - 1) / kPage;
  const int A = (sink + kPage - 1) / kPage;             // pages holding sink tokens
  const int Bp = max(A, rstart / kPage);                // first further page holding recent ones
  const int nwin = A + (n_pages - Bp);
  const int32_t* ptab = a.bf16_page_table + static_cast<size_t>(b) * a.max_pages;

  uint32_t qf[16];
  bf16_q_frags(a, b, kv, g, t, qf);
  float acc[8][4];
#pragma unroll
  for (int mb = 0; mb < 8; ++mb)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[mb][k] = 0.0f;
  float m_run = -INFINITY, l_run = 0.0f;
  for (int i = warp; i < nwin; i += kCombineWarps) {
    const int pg = i < A ? i : Bp + (i - A);
    const int id = ptab[pg];
    if (id < 0 || id >= a.bf16_num_pool_pages) {
      if (lane == 0) atomicOr(a.status, KVQ_STATUS_BAD_PAGE);
      continue;
    }
    const uint8_t* rec = a.bf16_pool + (static_cast<size_t>(id) * a.Hkv + kv) * kBf16Rec;
    uint4 vf[8];
#pragma unroll
    for (int mb = 0; mb < 8; ++mb)
      vf[mb] = __ldg(reinterpret_cast<const uint4*>(rec + 4096 + 512 * mb + 16 * lane));
    float s[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const uint4 kf = __ldg(reinterpret_cast<const uint4*>(rec + 512 * w + 16 * lane));
      mma_bf16(s, kf.x, kf.y, kf.z, kf.w, qf[2 * w], qf[2 * w + 1]);
    }
    const int pos0 = pg * kPage + g, pos1 = pos0 + 8;
    const bool v0 = pos0 < len && (pos0 < sink || pos0 >= rstart);
    const bool v1 = pos1 < len && (pos1 < sink || pos1 >= rstart);
    bf16_page_update(s, vf, v0, v1, a.log2_scale, g, t, acc, m_run, l_run);
  }
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) l_run += __shfl_xor_sync(0xffffffffu, l_run, off);
  if (t < a.G) {
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) {
      ws.o[warp][t][16 * mb + g] = acc[mb][0] + acc[mb][1];
      ws.o[warp][t][16 * mb + g + 8] = acc[mb][2] + acc[mb][3];
    }
    if (g == 0) {
      ws.m[warp][t] = m_run;
      ws.l[warp][t] = l_run;
    }
  }
  __syncthreads();
  const int h = tid / kDim, d = tid % kDim;
  float o = 0.0f;
  if (h < a.G) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) M = fmaxf(M, ws.m[w][h]);
    float L = 0.0f;
    if (M > -INFINITY) {
#pragma unroll 4
      for (int w = 0; w < kCombineWarps; ++w) {
        if (ws.m[w][h] == -INFINITY) continue;
        const float f = fast_exp2(ws.m[w][h] - M);
        L = fmaf(f, ws.l[w][h], L);
        o = fmaf(f, ws.o[w][h][d], o);
      }
    }
    if (d == 0) {
      ws.M[h] = M;
      ws.L[h] = L;
    }
  }
  return o;
}

template <bool kWindow>
__global__ void __launch_bounds__(kCombineThreads, 1) combine_kernel(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  CombineSmem& sm = *reinterpret_cast<CombineSmem*>(smem_raw);
  WindowSmem& ws = *reinterpret_cast<WindowSmem*>(smem_raw + sizeof(CombineSmem));
  const int b = blockIdx.x, kv = blockIdx.y, tid = threadIdx.x;
  const int h = tid / kDim, d = tid % kDim;       // thread (h, d)
  const int warp = tid >> 5, lane = tid & 31;
  int S = a.splits;
  const int G = a.G;
  const uint32_t bar = smem_u32(&sm.bar);
  // Let the next kernel in the stream launch now: the kernels of this library
  // read nothing this one writes before their own griddepcontrol.wait, so the
  // next decode step can stage its rotation matrices while this merge runs.
  griddep_launch_dependents();
  // the matrix of the one basis change: R_V^T (INT2 part back to the plain
  // basis) or, for a rotated-basis output, R_V (window part forward)
  const bool stage = kWindow || a.rotate_out;
  if (stage && tid == 0) {
    const float* R = a.rotate_out ? a.RVt : a.RV;
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, kDim * kDim * 4);
    bulk_g2s(smem_u32(sm.Rt), R + static_cast<size_t>(kv) * kDim * kDim, kDim * kDim * 4, bar);
  }
  float owin = 0.0f;
  if constexpr (kWindow) owin = window_partial(a, ws, b, kv);
  griddep_wait();       // the partials come from the decode kernel
  // balanced schedule: sequence b's splits are partial slots sched_base[b] ...
  // (all heads of a slot side by side); otherwise b's splits of a head are adjacent
  int pbase = 0;
  if (a.balanced) {
    S = a.sched_nsplit[b];
    pbase = a.sched_base[b];
  }
  const int pstride = a.balanced ? a.H * kPartStride : kPartStride;   // floats between splits
  auto head_parts = [&](int head) -> const float* {
    return a.balanced ? a.part + (static_cast<size_t>(pbase) * a.H + head) * kPartStride
                      : a.part + (static_cast<size_t>(b) * a.H + head) * a.splits * kPartStride;
  };
  // Thread (h, d) loads element d of its head's first kPre split partials now,
  // so that these loads and the (m, l) loads below share one round trip.
  constexpr int kPre = 48;
  const float* parts_h = head_parts(kv * G + h);
  float v[kPre];
#pragma unroll
  for (int u = 0; u < kPre; ++u) v[u] = (h < G && u < S) ? parts_h[u * pstride + 4 + d] : 0.0f;
  if (kWindow) __syncthreads();   // ws.M / ws.L
  if (warp < G) {
    const float* parts = head_parts(kv * G + warp);
    // INT2 logits were taken against centred keys: with a window, add q.mu back
    const float qmu =
        kWindow ? a.qmeta[(static_cast<size_t>(b) * a.Hkv + kv) * kQMeta + 8 + warp] : 0.0f;
    // (m, l) of splits lane and lane + 32 in the same round trip as the
    // partials above; only splits beyond 64 are read by a second one
    constexpr int kML = 2;
    float mk[kML], lk[kML];
#pragma unroll
    for (int k = 0; k < kML; ++k) {
      const int j = lane + 32 * k;
      mk[k] = j < S ? parts[j * pstride] : -INFINITY;
      lk[k] = j < S ? parts[j * pstride + 1] : 0.0f;
    }
    float M = fmaxf(mk[0], mk[1]);
    for (int j = lane + 32 * kML; j < S; j += 32) M = fmaxf(M, parts[j * pstride]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    if (kWindow) M = fmaxf(M + qmu, ws.M[warp]);
    float L = 0.0f;
#pragma unroll
    for (int k = 0; k < kML; ++k) {
      const int j = lane + 32 * k;
      if (j < S) {
        const float w = (mk[k] == -INFINITY) ? 0.0f : fast_exp2(mk[k] + qmu - M);
        sm.w[warp][j] = w;
        L = fmaf(w, lk[k], L);
      }
    }
    for (int j = lane + 32 * kML; j < S; j += 32) {
      const float mj = parts[j * pstride];
      const float lj = parts[j * pstride + 1];
      const float w = (mj == -INFINITY) ? 0.0f : fast_exp2(mj + qmu - M);
      sm.w[warp][j] = w;
      L = fmaf(w, lj, L);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    if (lane == 0) {
      if (kWindow) {
        const float ww = (ws.M[warp] == -INFINITY) ? 0.0f : fast_exp2(ws.M[warp] - M);
        sm.ww[warp] = ww;
        L = fmaf(ww, ws.L[warp], L);
      }
      sm.linv[warp] = (L > 0.0f) ? 1.0f / L : 0.0f;
    }
  }
  __syncthreads();
  float o = 0.0f;
  if (h < G) {
    // splits in order: the preloaded ones, then the rest kPre at a time
#pragma unroll
    for (int u = 0; u < kPre; ++u)
      if (u < S) o = fmaf(sm.w[h][u], v[u], o);
    for (int j0 = kPre; j0 < S; j0 += kPre) {
#pragma unroll
      for (int u = 0; u < kPre; ++u) v[u] = j0 + u < S ? parts_h[(j0 + u) * pstride + 4 + d] : 0.0f;
#pragma unroll
      for (int u = 0; u < kPre; ++u)
        if (j0 + u < S) o = fmaf(sm.w[h][j0 + u], v[u], o);
    }
    if (!kWindow) o *= sm.linv[h];
  }
  if (stage) {
    // y R for the part that changes basis; thread (q, d) sums j in quarter q
    // for every head, so each element of the matrix is read once per CTA
    sm.ot[d][h] = (kWindow && !a.rotate_out) ? owin : o;
    const bool ok = mbar_wait_bounded(bar, 0);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        atomicOr(a.status, KVQ_STATUS_TIMEOUT);
        mbar_drain(bar, 0);
      }
      return;
    }
    {
      const int q = h;
      float r4[kMaxG] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 8
      for (int jj = 0; jj < kDim / 4; ++jj) {
        const int j = q * (kDim / 4) + jj;
        const float4 ov = *reinterpret_cast<const float4*>(sm.ot[j]);
        const float rt = sm.Rt[j * kDim + d];
        r4[0] = fmaf(ov.x, rt, r4[0]);
        r4[1] = fmaf(ov.y, rt, r4[1]);
        r4[2] = fmaf(ov.z, rt, r4[2]);
        r4[3] = fmaf(ov.w, rt, r4[3]);
      }
#pragma unroll
      for (int hh = 0; hh < kMaxG; ++hh) sm.red[q][hh][d] = r4[hh];
    }
    __syncthreads();
    const float r = (sm.red[0][h][d] + sm.red[1][h][d]) + (sm.red[2][h][d] + sm.red[3][h][d]);
    if (!kWindow) o = r;
    else if (h < G) o = (a.rotate_out ? fmaf(sm.ww[h], owin, r) : fmaf(sm.ww[h], r, o)) * sm.linv[h];
  }
  if (h < G) a.out[(static_cast<size_t>(b) * a.H + kv * G + h) * kDim + d] = o;
}

// The KV-head combine in 256-thread CTAs (four per SM, so that a batch of up
// to 4 x #SMs (sequence, KV head) pairs takes one wave), with the same
// arithmetic in the same order as combine_kernel<false>.  Merge: the two warps
// of head h = tid / 64 each compute the head's (m, l) weights over the splits
// (lane j holds splits j and j + 32) and thread (h, p) merges elements 2p and
// 2p + 1, taking each weight from its lane by a shuffle, so no barrier
// separates the weights from the merge.  Basis change: R_V^T is read from
// global memory (L2) rather than staged, thread (q, p) = (tid / 64, tid % 64)
// sums quarter q of j for elements 2p, 2p + 1 of all G heads.
constexpr int kC4Threads = 256;
constexpr int kC4Pre = 12;
struct Combine4Smem {
  alignas(16) float ot[kDim][kMaxG];   // the G merged outputs, element-major
  float red[4][kMaxG][kDim];           // per-quarter sums of the basis change
};

__global__ void __launch_bounds__(kC4Threads, 4) combine4_kernel(DecodeArgs a) {
  __shared__ Combine4Smem sm;
  const int b = blockIdx.x, kv = blockIdx.y, tid = threadIdx.x;
  const int lane = tid & 31;
  const int G = a.G;
  griddep_launch_dependents();
  griddep_wait();       // the partials come from the decode kernel
  int S = a.splits, pbase = 0;
  if (a.balanced) {
    S = a.sched_nsplit[b];
    pbase = a.sched_base[b];
  }
  const int pstride = a.balanced ? a.H * kPartStride : kPartStride;
  const int h = tid >> 6, p = tid & 63;
  const bool live = h < G;              // uniform across each warp
  float2 o = make_float2(0.0f, 0.0f);
  if (live) {
    const float* parts =
        a.balanced ? a.part + (static_cast<size_t>(pbase) * a.H + kv * G + h) * kPartStride
                   : a.part + (static_cast<size_t>(b) * a.H + kv * G + h) * a.splits * kPartStride;
    const float* pv = parts + 4 + 2 * p;
    // the first kC4Pre partials and the (m, l) of splits lane, lane + 32 in one
    // round trip
    float2 v[kC4Pre];
#pragma unroll
    for (int k = 0; k < kC4Pre; ++k)
      v[k] = k < S ? *reinterpret_cast<const float2*>(pv + k * pstride) : make_float2(0.0f, 0.0f);
    float mk[2], lk[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int j = lane + 32 * k;
      mk[k] = j < S ? parts[j * pstride] : -INFINITY;
      lk[k] = j < S ? parts[j * pstride + 1] : 0.0f;
    }
    float M = fmaxf(mk[0], mk[1]);
    for (int j = lane + 64; j < S; j += 32) M = fmaxf(M, parts[j * pstride]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float wk[2];
    float L = 0.0f;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int j = lane + 32 * k;
      wk[k] = (j < S && mk[k] != -INFINITY) ? fast_exp2(mk[k] - M) : 0.0f;
      if (j < S) L = fmaf(wk[k], lk[k], L);
    }
    for (int j = lane + 64; j < S; j += 32) {
      const float mj = parts[j * pstride];
      const float lj = parts[j * pstride + 1];
      const float w = (mj == -INFINITY) ? 0.0f : fast_exp2(mj - M);
      L = fmaf(w, lj, L);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    const float linv = (L > 0.0f) ? 1.0f / L : 0.0f;
    // weight of split j: lane j % 32 of wk[j / 32] (recomputed past 64 splits)
    auto weight = [&](int j) -> float {
      if (j < 64) return __shfl_sync(0xffffffffu, j < 32 ? wk[0] : wk[1], j & 31);
      const float mj = parts[j * pstride];
      return (mj == -INFINITY) ? 0.0f : fast_exp2(mj - M);
    };
#pragma unroll
    for (int k = 0; k < kC4Pre; ++k) {
      if (k < S) {
        const float w = weight(k);
        o.x = fmaf(w, v[k].x, o.x);
        o.y = fmaf(w, v[k].y, o.y);
      }
    }
    for (int j0 = kC4Pre; j0 < S; j0 += kC4Pre) {
#pragma unroll
      for (int k = 0; k < kC4Pre; ++k)
        v[k] = j0 + k < S ? *reinterpret_cast<const float2*>(pv + (j0 + k) * pstride)
                          : make_float2(0.0f, 0.0f);
#pragma unroll
      for (int k = 0; k < kC4Pre; ++k) {
        if (j0 + k < S) {
          const float w = weight(j0 + k);
          o.x = fmaf(w, v[k].x, o.x);
          o.y = fmaf(w, v[k].y, o.y);
        }
      }
    }
    o.x *= linv;
    o.y *= linv;
  }
  float* out = a.out + (static_cast<size_t>(b) * a.H + kv * G + h) * kDim + 2 * p;
  if (!a.rotate_out) {
    if (live) *reinterpret_cast<float2*>(out) = o;
    return;
  }
  sm.ot[2 * p][h] = o.x;
  sm.ot[2 * p + 1][h] = o.y;
  __syncthreads();
  {
    const int q = tid >> 6;
    const float* Rt = a.RVt + static_cast<size_t>(kv) * kDim * kDim + 2 * p;
    float r[kMaxG][2];
#pragma unroll
    for (int hh = 0; hh < kMaxG; ++hh) r[hh][0] = r[hh][1] = 0.0f;
#pragma unroll 8
    for (int jj = 0; jj < kDim / 4; ++jj) {
      const int j = q * (kDim / 4) + jj;
      const float4 ov = *reinterpret_cast<const float4*>(sm.ot[j]);
      const float2 rt = __ldg(reinterpret_cast<const float2*>(Rt + j * kDim));
      r[0][0] = fmaf(ov.x, rt.x, r[0][0]);
      r[0][1] = fmaf(ov.x, rt.y, r[0][1]);
      r[1][0] = fmaf(ov.y, rt.x, r[1][0]);
      r[1][1] = fmaf(ov.y, rt.y, r[1][1]);
      r[2][0] = fmaf(ov.z, rt.x, r[2][0]);
      r[2][1] = fmaf(ov.z, rt.y, r[2][1]);
      r[3][0] = fmaf(ov.w, rt.x, r[3][0]);
      r[3][1] = fmaf(ov.w, rt.y, r[3][1]);
    }
#pragma unroll
    for (int hh = 0; hh < kMaxG; ++hh) {
      sm.red[q][hh][2 * p] = r[hh][0];
      sm.red[q][hh][2 * p + 1] = r[hh][1];
    }
  }
  __syncthreads();
  if (live) {
    float2 y;
    y.x = (sm.red[0][h][2 * p] + sm.red[1][h][2 * p]) + (sm.red[2][h][2 * p] + sm.red[3][h][2 * p]);
    y.y = (sm.red[0][h][2 * p + 1] + sm.red[1][h][2 * p + 1]) +
          (sm.red[2][h][2 * p + 1] + sm.red[3][h][2 * p + 1]);
    *reinterpret_cast<float2*>(out) = y;
  }
}

// The same combine with one CTA per query head (b, kv, h), for calls whose
// (sequence, query head) count fills at most one wave of these CTAs (short
// contexts with many splits, such as a 36-layer stack at 8K): each CTA merges
// one head, so the partials a CTA loads and the dependent steps before its
// store are a quarter of the per-KV-head combine's.  Thread (qq, d), qq =
// tid / 128: element d of splits qq, qq + 4, ... (four interleaved quarters of
// the merge, added in a fixed order), then quarter qq of the basis change of
// element d.  R_V^T is staged by a bulk copy issued before the dependency wait.
struct HeadCombineSmem {
  float Rt[kDim * kDim];
  float w[kMaxSplits];
  float red[4][kDim];
  float o[kDim];
  float linv;
  uint64_t bar;
};
constexpr int kHeadCombineCtasPerSm = 2;

__global__ void __launch_bounds__(kCombineThreads, kHeadCombineCtasPerSm)
    combine_head_kernel(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  HeadCombineSmem& sm = *reinterpret_cast<HeadCombineSmem*>(smem_raw);
  const int b = blockIdx.x, kv = blockIdx.y, h = blockIdx.z, tid = threadIdx.x;
  const int qq = tid / kDim, d = tid % kDim;
  const int warp = tid >> 5, lane = tid & 31;
  int S = a.splits;
  const int G = a.G;
  const uint32_t bar = smem_u32(&sm.bar);
  griddep_launch_dependents();      // as in combine_kernel
  const bool stage = a.rotate_out != 0;
  if (stage && tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, kDim * kDim * 4);
    bulk_g2s(smem_u32(sm.Rt), a.RVt + static_cast<size_t>(kv) * kDim * kDim, kDim * kDim * 4, bar);
  }
  griddep_wait();       // the partials come from the decode kernel
  // balanced schedule: sequence b's splits are partial slots sched_base[b] ...
  // (all heads of a slot side by side); otherwise b's splits of a head are adjacent
  int pbase = 0;
  if (a.balanced) {
    S = a.sched_nsplit[b];
    pbase = a.sched_base[b];
  }
  const int pstride = a.balanced ? a.H * kPartStride : kPartStride;   // floats between splits
  auto head_parts = [&](int head) -> const float* {
    return a.balanced ? a.part + (static_cast<size_t>(pbase) * a.H + head) * kPartStride
                      : a.part + (static_cast<size_t>(b) * a.H + head) * a.splits * kPartStride;
  };
  const float* parts = head_parts(kv * G + h);
  constexpr int kPreQ = 16;         // splits qq + 4u, u < kPreQ, loaded in the first round trip
  float v[kPreQ];
#pragma unroll
  for (int u = 0; u < kPreQ; ++u) {
    const int s = qq + 4 * u;
    v[u] = s < S ? parts[s * pstride + 4 + d] : 0.0f;
  }
  if (warp == 0) {
    constexpr int kML = 2;
    float mk[kML], lk[kML];
#pragma unroll
    for (int k = 0; k < kML; ++k) {
      const int j = lane + 32 * k;
      mk[k] = j < S ? parts[j * pstride] : -INFINITY;
      lk[k] = j < S ? parts[j * pstride + 1] : 0.0f;
    }
    float M = fmaxf(mk[0], mk[1]);
    for (int j = lane + 32 * kML; j < S; j += 32) M = fmaxf(M, parts[j * pstride]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.0f;
#pragma unroll
    for (int k = 0; k < kML; ++k) {
      const int j = lane + 32 * k;
      if (j < S) {
        const float w = (mk[k] == -INFINITY) ? 0.0f : fast_exp2(mk[k] - M);
        sm.w[j] = w;
        L = fmaf(w, lk[k], L);
      }
    }
    for (int j = lane + 32 * kML; j < S; j += 32) {
      const float mj = parts[j * pstride];
      const float lj = parts[j * pstride + 1];
      const float w = (mj == -INFINITY) ? 0.0f : fast_exp2(mj - M);
      sm.w[j] = w;
      L = fmaf(w, lj, L);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    if (lane == 0) sm.linv = (L > 0.0f) ? 1.0f / L : 0.0f;
  }
  __syncthreads();
  float o = 0.0f;
#pragma unroll
  for (int u = 0; u < kPreQ; ++u)
    if (qq + 4 * u < S) o = fmaf(sm.w[qq + 4 * u], v[u], o);
  for (int s0 = 4 * kPreQ; s0 < S; s0 += 4 * kPreQ) {
#pragma unroll
    for (int u = 0; u < kPreQ; ++u) {
      const int s = s0 + qq + 4 * u;
      v[u] = s < S ? parts[s * pstride + 4 + d] : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < kPreQ; ++u)
      if (s0 + qq + 4 * u < S) o = fmaf(sm.w[s0 + qq + 4 * u], v[u], o);
  }
  sm.red[qq][d] = o;
  __syncthreads();
  if (qq == 0)
    sm.o[d] = ((sm.red[0][d] + sm.red[1][d]) + (sm.red[2][d] + sm.red[3][d])) * sm.linv;
  float* out = a.out + (static_cast<size_t>(b) * a.H + kv * G + h) * kDim;
  if (!stage) {
    if (qq == 0) out[d] = sm.o[d];
    return;
  }
  const bool ok = mbar_wait_bounded(bar, 0);
  if (__syncthreads_or(!ok)) {      // also orders sm.o and sm.red before the reuse below
    if (tid == 0) {
      atomicOr(a.status, KVQ_STATUS_TIMEOUT);
      mbar_drain(bar, 0);
    }
    return;
  }
  // y R_V^T: thread (qq, d) sums j in quarter qq
  float r = 0.0f;
#pragma unroll 8
  for (int jj = 0; jj < kDim / 4; ++jj) {
    const int j = qq * (kDim / 4) + jj;
    r = fmaf(sm.o[j], sm.Rt[j * kDim + d], r);
  }
  sm.red[qq][d] = r;
  __syncthreads();
  if (qq == 0) out[d] = (sm.red[0][d] + sm.red[1][d]) + (sm.red[2][d] + sm.red[3][d]);
}

// Dequantise positions [start, start+len) of one sequence: CTA per (position,
// KV head), thread d per element, following the record layout of include/kvq.h.
__global__ void __launch_bounds__(128) dequant_kernel(const uint8_t* __restrict__ pool,
                                                      int num_pool_pages,
                                                      const int32_t* __restrict__ page_table,
                                                      int max_pages, int Hkv, int seq, int start,
                                                      float* K_out, float* V_out,
                                                      uint32_t* status) {
  const int i = blockIdx.x, kv = blockIdx.y, d = threadIdx.x;
  const int p = start + i;
  if (p < 0 || p >= max_pages * kPage) {
    if (d == 0) atomicOr(status, KVQ_STATUS_BAD_POS);
    return;
  }
  const int id = page_table[static_cast<size_t>(seq) * max_pages + p / kPage];
  if (id < 0 || id >= num_pool_pages) {
    if (d == 0) atomicOr(status, KVQ_STATUS_BAD_PAGE);
    return;
  }
  const uint8_t* rec = pool + (static_cast<size_t>(id) * Hkv + kv) * kInt2Rec;
  const uint32_t* words = reinterpret_cast<const uint32_t*>(rec);
  const int tau = p % kPage;
  const size_t o = (static_cast<size_t>(i) * Hkv + kv) * kDim + d;
  if (K_out) {
    const int w = d >> 4, r = d & 15, h = r >> 3, t = (r >> 1) & 3, e = r & 1;
    const int L = 4 * (tau & 7) + t, word = 2 * (tau >> 3) + h, bit = 16 * e + 2 * w;
    const uint32_t code = (words[4 * L + word] >> bit) & 3u;
    const uint32_t sz = *reinterpret_cast<const uint32_t*>(rec + 1024 + 16 * (tau & 7) + 4 * (tau >> 3));
    K_out[o] = fmaf(static_cast<float>(code), half_lo(sz), half_hi(sz));
  }
  if (V_out) {
    const int m = d >> 4, r = d & 15, g = r & 7, dh = r >> 3;
    const int t = (tau & 7) >> 1, e = tau & 1, th = tau >> 3;
    const int L = 4 * g + t, word = 2 * th + dh, bit = 16 * e + 2 * m;
    const uint32_t code = (words[128 + 4 * L + word] >> bit) & 3u;
    const uint32_t sz =
        *reinterpret_cast<const uint32_t*>(rec + 1024 + 16 * (tau & 7) + 8 + 4 * (tau >> 3));
    V_out[o] = fmaf(static_cast<float>(code), half_lo(sz), half_hi(sz));
  }
}

// out[c][j][i] = in[c][i][j] for count 128x128 matrices.
__global__ void transpose_kernel(const float* __restrict__ in, float* __restrict__ out) {
  __shared__ float tile[32][33];
  const float* src = in + static_cast<size_t>(blockIdx.z) * kDim * kDim;
  float* dst = out + static_cast<size_t>(blockIdx.z) * kDim * kDim;
  const int bx = blockIdx.x * 32, by = blockIdx.y * 32;
  for (int k = threadIdx.y; k < 32; k += blockDim.y)
    tile[k][threadIdx.x] = src[(by + k) * kDim + bx + threadIdx.x];
  __syncthreads();
  for (int k = threadIdx.y; k < 32; k += blockDim.y)
    dst[(bx + k) * kDim + by + threadIdx.x] = tile[threadIdx.x][k];
}

// Dynamic shared-memory size and carve-out of kernel kKern, set once per
// device (one flag set per kernel: each instantiation of this template is
// its own kernel).
template <typename Smem, auto kKern>
cudaError_t set_smem_attr() {
  static bool done[64] = {};
  const auto kern = kKern;
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(sizeof(Smem)));
  // as much of the L1/shared split as possible for shared memory (two INT2
  // decode CTAs take 221 KB)
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             static_cast<int>(cudaSharedmemCarveoutMaxShared));
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

// Launch as a programmatic dependent of the preceding kernel in the stream.
template <typename... Args>
cudaError_t launch_dependent(void (*kern)(Args...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace

template <int NB>
cudaError_t launch_qprep_nb(const DecodeArgs& a, const float* RK, const float* mu, float sm_scale,
                            cudaStream_t st) {
  cudaError_t e = set_smem_attr<QprepSmem<NB>, qprep_kernel<NB>>();
  if (e != cudaSuccess) return e;
  dim3 grid((a.batch + NB - 1) / NB + (a.balanced ? 1 : 0), a.Hkv);
  e = launch_dependent(qprep_kernel<NB>, grid, dim3(128), sizeof(QprepSmem<NB>), st, a, RK, mu,
                       sm_scale * kLog2e);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_qprep(const DecodeArgs& a, const float* RK, const float* mu, float sm_scale,
                         cudaStream_t st) {
  // the query groups of the step preparation with the same prep_nb
  if (a.prep_nb >= 2) return launch_qprep_nb<2>(a, RK, mu, sm_scale, st);
  return launch_qprep_nb<1>(a, RK, mu, sm_scale, st);
}

template <int NB>
cudaError_t launch_step_prep_nb(const DecodeArgs& a, const StepArgs& sa, cudaStream_t st) {
  cudaError_t e = set_smem_attr<StepPrepSmem<NB>, step_prep_kernel<NB>>();
  if (e != cudaSuccess) return e;
  e = launch_dependent(step_prep_kernel<NB>,
                       dim3((a.batch + NB - 1) / NB + (a.balanced ? 1 : 0), a.Hkv, step_roles<NB>()),
                       dim3(128),
                       sizeof(StepPrepSmem<NB>), st, a, sa);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_step_prep(const DecodeArgs& a, const StepArgs& sa, cudaStream_t st) {
  if (a.prep_nb >= 8) return launch_step_prep_nb<8>(a, sa, st);
  if (a.prep_nb >= 4) return launch_step_prep_nb<4>(a, sa, st);
  if (a.prep_nb == 2) return launch_step_prep_nb<2>(a, sa, st);
  return launch_step_prep_nb<1>(a, sa, st);
}

cudaError_t launch_decode_int2(const DecodeArgs& a, cudaStream_t st) {
  cudaError_t e;
  if (a.balanced) {
    e = set_smem_attr<Int2Smem, decode_int2_kernel<true>>();
    if (e != cudaSuccess) return e;
    e = launch_dependent(decode_int2_kernel<true>, dim3(a.batch * a.splits, a.Hkv / a.hpc, 1),
                         dim3(kW * 32), sizeof(Int2Smem), st, a);
  } else {
    e = set_smem_attr<Int2Smem, decode_int2_kernel<false>>();
    if (e != cudaSuccess) return e;
    e = launch_dependent(decode_int2_kernel<false>, dim3(a.splits, a.Hkv / a.hpc, a.batch),
                         dim3(kW * 32), sizeof(Int2Smem), st, a);
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_decode_bf16(const DecodeArgs& a, cudaStream_t st) {
  cudaError_t e = set_smem_attr<Bf16Smem, decode_bf16_kernel>();
  if (e != cudaSuccess) return e;
  dim3 grid(a.splits, a.Hkv, a.batch);
  e = launch_dependent(decode_bf16_kernel, grid, dim3(kDecodeThreads), sizeof(Bf16Smem), st, a);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_combine(const DecodeArgs& a, cudaStream_t st) {
  cudaError_t e;
  if (a.window) {
    e = set_smem_attr<CombineWindowSmem, combine_kernel<true>>();
    if (e != cudaSuccess) return e;
    e = launch_dependent(combine_kernel<true>, dim3(a.batch, a.Hkv), dim3(kCombineThreads),
                         sizeof(CombineWindowSmem), st, a);
  } else if (a.combine_per_head) {
    e = set_smem_attr<HeadCombineSmem, combine_head_kernel>();
    if (e != cudaSuccess) return e;
    e = launch_dependent(combine_head_kernel, dim3(a.batch, a.Hkv, a.G), dim3(kCombineThreads),
                         sizeof(HeadCombineSmem), st, a);
  } else if (a.combine_small) {
    e = launch_dependent(combine4_kernel, dim3(a.batch, a.Hkv), dim3(kC4Threads), 0, st, a);
  } else {
    e = set_smem_attr<CombineSmem, combine_kernel<false>>();
    if (e != cudaSuccess) return e;
    e = launch_dependent(combine_kernel<false>, dim3(a.batch, a.Hkv), dim3(kCombineThreads),
                         sizeof(CombineSmem), st, a);
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_dequant(const uint8_t* pool, int num_pool_pages, const int32_t* page_table,
                           int max_pages, int Hkv, int seq, int start, int len, float* K_out,
                           float* V_out, uint32_t* status, cudaStream_t st) {
  dim3 grid(len, Hkv);
  dequant_kernel<<<grid, 128, 0, st>>>(pool, num_pool_pages, page_table, max_pages, Hkv, seq,
                                       start, K_out, V_out, status);
  return cudaGetLastError();
}

cudaError_t launch_transpose(const float* in, float* out, int count, cudaStream_t st) {
  dim3 grid(kDim / 32, kDim / 32, count), block(32, 8);
  transpose_kernel<<<grid, block, 0, st>>>(in, out);
  return cudaGetLastError();
}

int combine_head_ctas_per_sm() { return kHeadCombineCtasPerSm; }

template <int NB>
static int step_prep_ctas_per_sm_nb() {
  if (set_smem_attr<StepPrepSmem<NB>, step_prep_kernel<NB>>() != cudaSuccess) return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, step_prep_kernel<NB>, 128,
                                                    sizeof(StepPrepSmem<NB>)) != cudaSuccess ||
      n < 1)
    return 1;
  return n;
}

int step_prep_ctas_per_sm(int nb) {
  switch (nb) {
    case 8: return step_prep_ctas_per_sm_nb<8>();
    case 4: return step_prep_ctas_per_sm_nb<4>();
    case 2: return step_prep_ctas_per_sm_nb<2>();
    default: return step_prep_ctas_per_sm_nb<1>();
  }
}

int decode_int2_ctas_per_sm() {
  if (set_smem_attr<Int2Smem, decode_int2_kernel<false>>() != cudaSuccess) return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_int2_kernel<false>, kW * 32,
                                                    sizeof(Int2Smem)) != cudaSuccess || n < 1)
    return 1;
  return n;
}

int decode_bf16_ctas_per_sm() {
  if (set_smem_attr<Bf16Smem, decode_bf16_kernel>() != cudaSuccess) return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_bf16_kernel, kDecodeThreads,
                                                    sizeof(Bf16Smem)) != cudaSuccess || n < 1)
    return 1;
  return n;
}

}  // namespace kvq
