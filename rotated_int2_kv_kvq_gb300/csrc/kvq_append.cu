// kvq_append.cu — quantise-on-append into the paged INT2 cache, and the plain
// copy into the BF16 comparison cache.
//
// Method: "Output-Aware Rotation for INT2 KV-Cache Quantization" (pith.science
// review of arXiv 2608.02691), "What carries the argument": keys are centred by
// a per-channel mean (mechanism 2), then rotated, clipped, grouped and rounded
// to INT2 (mechanism 3); clip ratios c_K, c_V from "Assumptions & free
// parameters".  The integer format (asymmetric, one group of 128 per token,
// fp16 scale/zero) and the fp32 operation sequence are this library's, written
// out in include/kvq.h.  Every operation below whose rounding matters is an
// explicit round-to-nearest intrinsic (__fsub_rn, __fmul_rn, __fdiv_rn, fmaf),
// so the compiler cannot contract or reorder it and the stored bytes are
// reproducible bit for bit.
#include "kvq_internal.cuh"

namespace kvq {
namespace {

constexpr int kRBytes = kDim * kDim * 4;   // one rotation matrix in fp32
constexpr int kAUnroll = 8;                // rotation steps unrolled
// A token's 128 codes (one byte each) take a row of 132 bytes: rows 33 words
// apart put the eight tokens that a warp's lanes read together in eight
// different banks during the scatter.
constexpr int kCodeRow = kDim + 4;

// code = min(max(rint(fl(d / s)), 0), 3), fl the correctly rounded fp32
// quotient, for s > 0.  The quotient is first taken as d * rcp(s) (rcp.approx:
// relative error below 2^-22, the product's rounding 2^-24): for |q| < 4 that
// estimate is within 2^-20 of d / s, and fl(d / s) within 2^-23, so unless the
// estimate lies within 2^-18 of a half-integer both round to the same integer
// and the estimate decides the code.  Otherwise (rare) the correctly rounded
// division decides it, as the format's operation sequence states.  For
// |q| >= 4 both clamp to 3 (or 0), NaN gives 0 either way.
__device__ __forceinline__ float rcp_approx(float s) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
  return r;
}
// max / min over the warp's 32 lanes in one instruction (NaN inputs ignored,
// like fmaxf / fminf)
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float warp_min(float v) {
  float r;
  asm volatile("redux.sync.min.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ uint32_t clamp_code(float q) {
  return static_cast<uint32_t>(fminf(fmaxf(rintf(q), 0.0f), 3.0f));
}
__device__ __forceinline__ bool near_half(float q) {
  return fabsf(__fsub_rn(__fsub_rn(q, floorf(q)), 0.5f)) < 0x1p-18f;
}

template <int TPW, int NW>
struct AppendSmem {
  static constexpr int kTile = NW * TPW;                        // tokens per tile
  static constexpr int kR = 0;                                  // float [128][128]
  static constexpr int kC = kR + kRBytes;                       // float [128][kTile]
  static constexpr int kCodes = kC + kDim * kTile * 4;          // u8 [kTile][kCodeRow]
  static constexpr int kMu = kCodes + kTile * kCodeRow;         // float [128]
  static constexpr int kSZ = kMu + kDim * 4;                    // u32 [kTile]
  static constexpr int kRec = kSZ + kTile * 4;                  // long long [kTile]
  static constexpr int kBar = kRec + kTile * 8;                 // mbarrier
  static constexpr int kBytes = kBar + 16;
};

__device__ __forceinline__ float bf16_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// Quantise tiles of tokens for one (KV head, K|V).  TPW = tokens per warp.
// Warp w owns tokens [w*TPW, (w+1)*TPW) of a tile; lane L owns output elements
// 4L..4L+3 of each of them.
template <int TPW, int NW>
__global__ void __launch_bounds__(NW * 32) append_int2_kernel(AppendArgs a) {
  constexpr int kAppThreads = NW * 32;
  using S = AppendSmem<TPW, NW>;
  constexpr int kTile = S::kTile;
  extern __shared__ __align__(128) uint8_t smem[];
  float* Rs = reinterpret_cast<float*>(smem + S::kR);
  float* Cs = reinterpret_cast<float*>(smem + S::kC);
  uint8_t* codes = smem + S::kCodes;
  float* mus = reinterpret_cast<float*>(smem + S::kMu);
  uint32_t* sz = reinterpret_cast<uint32_t*>(smem + S::kSZ);
  long long* rec = reinterpret_cast<long long*>(smem + S::kRec);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + S::kBar);

  const int kv = blockIdx.y;
  const int which = blockIdx.z;            // 0 keys, 1 values
  const float clip = which ? a.clip_v : a.clip_k;
  const float* R = a.R + (static_cast<size_t>(which) * a.Hkv + kv) * kDim * kDim;
  const float* mu = which ? nullptr : a.mu + static_cast<size_t>(kv) * kDim;
  const uint16_t* X = which ? a.V : a.K;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // A following decode call's query preparation reads neither the pool nor
  // this kernel's inputs: let it start now (it waits for this grid before it
  // finishes, so the decode kernel still sees every appended page).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // Stage this head's rotation matrix with one bulk copy.
  const uint32_t bar_a = smem_u32(bar);
  if (tid == 0) {
    mbar_init(bar_a, 1);
    fence_mbar_init();
  }
  for (int i = tid; i < kDim; i += kAppThreads) mus[i] = mu ? mu[i] : 0.0f;
  __syncthreads();
  if (tid == 0) {
    mbar_arrive_expect_tx(bar_a, kRBytes);
    bulk_g2s(smem_u32(Rs), R, kRBytes, bar_a);
  }
  bool r_ready = false;

  // The tile's tokens: 16-byte pieces (8 bf16) of [kTile][128], loaded one tile
  // ahead into registers so that the loads of tile i+1 are in flight while the
  // rotation of tile i runs.
  constexpr int kPieces = kTile * (kDim / 8);
  constexpr int kPre = (kPieces + kAppThreads - 1) / kAppThreads;
  uint4 pre[kPre];
  auto load_tile = [&](int t0) {
#pragma unroll
    for (int r = 0; r < kPre; ++r) {
      const int idx = tid + r * kAppThreads;
      const int k = idx % kTile, ch = idx / kTile;
      const int tok = t0 + k;
      pre[r] = make_uint4(0u, 0u, 0u, 0u);
      if (idx < kPieces && tok < a.n)
        pre[r] = *reinterpret_cast<const uint4*>(X + (static_cast<size_t>(tok) * a.Hkv + kv) * kDim +
                                                 ch * 8);
    }
  };
  if (static_cast<long long>(blockIdx.x) * kTile < a.n) load_tile(blockIdx.x * kTile);

  for (int tile = blockIdx.x; tile * kTile < a.n; tile += gridDim.x) {
    const int tok0 = tile * kTile;
    // (1) record address of each token of the tile (or -1 if it is skipped)
    if (tid < kTile) {
      const int tok = tok0 + tid;
      long long r = -1;
      if (tok < a.n) {
        const int b = a.seq_idx[tok];
        const int p = a.positions[tok];
        if (b < 0 || b >= a.batch) {
          atomicOr(a.status, KVQ_STATUS_BAD_SEQ);
        } else if (p < 0 || p >= a.max_pages * kPage) {
          atomicOr(a.status, KVQ_STATUS_BAD_POS);
        } else {
          const int page = a.page_table[static_cast<size_t>(b) * a.max_pages + p / kPage];
          if (page < 0 || page >= a.num_pool_pages) {
            atomicOr(a.status, KVQ_STATUS_BAD_PAGE);
          } else {
            r = ((static_cast<long long>(page) * a.Hkv + kv) * kInt2Rec) * kPage + (p % kPage);
          }
        }
      }
      rec[tid] = r;      // record byte offset * 16 + slot
    }
    // (2) the prefetched tile: centre keys (fp32 subtract), store transposed: Cs[j][k]
#pragma unroll
    for (int r = 0; r < kPre; ++r) {
      const int idx = tid + r * kAppThreads;
      if (idx < kPieces) {
        const int k = idx % kTile, ch = idx / kTile;
        const uint32_t w4[4] = {pre[r].x, pre[r].y, pre[r].z, pre[r].w};
        float v[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[2 * e] = bf16_to_f32(w4[e] & 0xffffu);
          v[2 * e + 1] = bf16_to_f32(w4[e] >> 16);
        }
        if (mu && tok0 + k < a.n) {
          const float4 m0 = *reinterpret_cast<const float4*>(mus + ch * 8);
          const float4 m1 = *reinterpret_cast<const float4*>(mus + ch * 8 + 4);
          const float mv[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) v[e] = __fsub_rn(v[e], mv[e]);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) Cs[(ch * 8 + e) * kTile + k] = v[e];
      }
    }
    if (!r_ready) {
      // every thread waits (bounded); the CTA leaves together if any gave up
      const bool ok = mbar_wait_bounded(bar_a, 0);
      if (__syncthreads_or(!ok)) {
        if (tid == 0) {
          atomicOr(a.status, KVQ_STATUS_TIMEOUT);
          mbar_drain(bar_a, 0);
        }
        return;      // nothing was written for this CTA
      }
      r_ready = true;
    }
    __syncthreads();
    // the next tile's tokens, in flight during this tile's rotation
    if (static_cast<long long>(tile + gridDim.x) * kTile < a.n) load_tile((tile + gridDim.x) * kTile);

    // (3) rotate: r_i = fmaf chain over j = 0..127 in order, for TPW tokens x 4 outputs
    float acc[TPW][4];
#pragma unroll
    for (int t = 0; t < TPW; ++t)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[t][c] = 0.0f;
    const float4* R4 = reinterpret_cast<const float4*>(Rs);
    const float* cw = Cs + warp * TPW;
    // operands of step j + 1 are loaded while step j's products run
    float4 rn = R4[lane];
    float cn[TPW];
    auto load_c = [&](int j, float (&c)[TPW]) {
      const float* cj = cw + j * kTile;
      if constexpr (TPW % 4 == 0) {
#pragma unroll
        for (int t = 0; t < TPW; t += 4) {
          const float4 c4 = *reinterpret_cast<const float4*>(cj + t);
          c[t] = c4.x; c[t + 1] = c4.y; c[t + 2] = c4.z; c[t + 3] = c4.w;
        }
      } else {
#pragma unroll
        for (int t = 0; t < TPW; ++t) c[t] = cj[t];
      }
    };
    load_c(0, cn);
#pragma unroll kAUnroll
    for (int j = 0; j < kDim; ++j) {
      const float4 r = rn;
      float c[TPW];
#pragma unroll
      for (int t = 0; t < TPW; ++t) c[t] = cn[t];
      if (j + 1 < kDim) {
        rn = R4[(j + 1) * (kDim / 4) + lane];
        load_c(j + 1, cn);
      }
#pragma unroll
      for (int t = 0; t < TPW; ++t) {
        acc[t][0] = fmaf(c[t], r.x, acc[t][0]);
        acc[t][1] = fmaf(c[t], r.y, acc[t][1]);
        acc[t][2] = fmaf(c[t], r.z, acc[t][2]);
        acc[t][3] = fmaf(c[t], r.w, acc[t][3]);
      }
    }

    // (4) group max/min (whole vector), clip, fp16 scale/zero, codes
#pragma unroll
    for (int t = 0; t < TPW; ++t) {
      const float mx = warp_max(fmaxf(fmaxf(acc[t][0], acc[t][1]), fmaxf(acc[t][2], acc[t][3])));
      const float mn = warp_min(fminf(fminf(acc[t][0], acc[t][1]), fminf(acc[t][2], acc[t][3])));
      const float mxc = __fmul_rn(clip, mx);
      const float mnc = __fmul_rn(clip, mn);
      const float s32 = __fdiv_rn(__fsub_rn(mxc, mnc), 3.0f);
      const __half sh = __float2half_rn(s32);
      const __half zh = __float2half_rn(mnc);
      const float s = __half2float(sh), z = __half2float(zh);
      uint32_t packed = 0;
      if (s != 0.0f) {
        const float rs = rcp_approx(s);
        float d[4], q[4];
        bool near = false;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          d[c] = __fsub_rn(acc[t][c], z);
          q[c] = __fmul_rn(d[c], rs);
          near = near || near_half(q[c]);
        }
        if (near) {
#pragma unroll
          for (int c = 0; c < 4; ++c) q[c] = __fdiv_rn(d[c], s);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) packed |= clamp_code(q[c]) << (8 * c);
      }
      const int k = warp * TPW + t;
      reinterpret_cast<uint32_t*>(codes)[k * (kCodeRow / 4) + lane] = packed;
      if (lane == 0)
        sz[k] = static_cast<uint32_t>(__half_as_ushort(sh)) |
                (static_cast<uint32_t>(__half_as_ushort(zh)) << 16);
    }
    __syncthreads();

    // (5) scatter into the page records (layout in include/kvq.h)
    if (which == 0) {
      // keys: per token, lane-group t of row (tau & 7): two adjacent words (h = 0, 1)
      for (int item = tid; item < kTile * 4; item += kAppThreads) {
        const int k = item >> 2, t = item & 3;
        const long long r = rec[k];
        if (r < 0) continue;
        const int tau = static_cast<int>(r % kPage);
        uint8_t* base = a.pool + r / kPage;
        const uint8_t* ck = codes + k * kCodeRow;
        uint32_t word[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t wv = 0;
#pragma unroll
          for (int w = 0; w < 8; ++w) {
            const int d = 16 * w + 2 * t + 8 * h;
            wv |= static_cast<uint32_t>(ck[d]) << (2 * w);
            wv |= static_cast<uint32_t>(ck[d + 1]) << (16 + 2 * w);
          }
          word[h] = wv;
        }
        const int L = 4 * (tau & 7) + t;
        *reinterpret_cast<uint2*>(base + 16 * L + 8 * (tau >> 3)) = make_uint2(word[0], word[1]);
      }
    } else {
      // values: per token, 8 lanes (g) x 2 words (dh), one 16-bit half each
      for (int item = tid; item < kTile * 16; item += kAppThreads) {
        const int k = item >> 4, g = (item >> 1) & 7, dh = item & 1;
        const long long r = rec[k];
        if (r < 0) continue;
        const int tau = static_cast<int>(r % kPage);
        uint8_t* base = a.pool + r / kPage;
        const uint8_t* ck = codes + k * kCodeRow;
        uint32_t hv = 0;
#pragma unroll
        for (int m = 0; m < 8; ++m) hv |= static_cast<uint32_t>(ck[16 * m + g + 8 * dh]) << (2 * m);
        const int t = (tau & 7) >> 1, e = tau & 1, th = tau >> 3;
        const int L = 4 * g + t;
        *reinterpret_cast<uint16_t*>(base + 512 + 16 * L + 4 * (2 * th + dh) + 2 * e) =
            static_cast<uint16_t>(hv);
      }
    }
    if (tid < kTile) {
      const long long r = rec[tid];
      if (r >= 0) {
        const int tau = static_cast<int>(r % kPage);
        uint8_t* base = a.pool + r / kPage;
        *reinterpret_cast<uint32_t*>(base + 1024 + 16 * (tau & 7) + (which ? 8 : 0) +
                                     4 * (tau >> 3)) = sz[tid];
      }
    }
    __syncthreads();   // Cs, codes, rec are rewritten by the next tile
  }
  if (!r_ready) {
    // no tile for this CTA: still let the staged copy land before exiting
    if (!mbar_wait_bounded(bar_a, 0)) {
      if (tid == 0) atomicOr(a.status, KVQ_STATUS_TIMEOUT);
      mbar_drain(bar_a, 0);
    }
  }
}

// BF16 comparison cache: store each element unchanged at its layout position.
// One CTA per (token, KV head); thread d handles element d of K and of V.
__global__ void __launch_bounds__(128) append_bf16_kernel(AppendArgs a) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tok = blockIdx.x, kv = blockIdx.y, d = threadIdx.x;
  const int b = a.seq_idx[tok];
  const int p = a.positions[tok];
  if (b < 0 || b >= a.batch) {
    if (d == 0) atomicOr(a.status, KVQ_STATUS_BAD_SEQ);
    return;
  }
  if (p < 0 || p >= a.max_pages * kPage) {
    if (d == 0) atomicOr(a.status, KVQ_STATUS_BAD_POS);
    return;
  }
  const int page = a.page_table[static_cast<size_t>(b) * a.max_pages + p / kPage];
  if (page < 0 || page >= a.num_pool_pages) {
    if (d == 0) atomicOr(a.status, KVQ_STATUS_BAD_PAGE);
    return;
  }
  uint8_t* base = a.pool + (static_cast<size_t>(page) * a.Hkv + kv) * kBf16Rec;
  const int tau = p % kPage;
  const size_t src = (static_cast<size_t>(tok) * a.Hkv + kv) * kDim + d;
  {
    const int w = d >> 4, r = d & 15, h = r >> 3, t = (r >> 1) & 3, e = r & 1;
    const int L = 4 * (tau & 7) + t, reg = (tau >> 3) + 2 * h;
    *reinterpret_cast<uint16_t*>(base + 512 * w + 16 * L + 4 * reg + 2 * e) = a.K[src];
  }
  {
    const int m = d >> 4, r = d & 15, g = r & 7, dh = r >> 3;
    const int t = (tau & 7) >> 1, e = tau & 1, th = tau >> 3;
    const int L = 4 * g + t, reg = 2 * th + dh;
    *reinterpret_cast<uint16_t*>(base + 4096 + 512 * m + 16 * L + 4 * reg + 2 * e) = a.V[src];
  }
}

template <int TPW, int NW>
cudaError_t launch_tpw(const AppendArgs& a, int num_sms, cudaStream_t st) {
  using S = AppendSmem<TPW, NW>;
  static bool attr_set[64] = {};       // per device: the attribute is per context
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(append_int2_kernel<TPW, NW>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, S::kBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const int tiles = (a.n + S::kTile - 1) / S::kTile;
  // One wave of CTAs (two per SM, the shared-memory limit); each CTA loops
  // over tiles so the rotation matrix is staged once per CTA, not once per
  // tile (measured: 408 us per 32,767-token prefill against 419 us with two
  // waves).
  const int per_head = a.Hkv * 2;
  int gx = (2 * num_sms + per_head - 1) / per_head;
  if (gx > tiles) gx = tiles;
  if (gx < 1) gx = 1;
  dim3 grid(gx, a.Hkv, 2);
  append_int2_kernel<TPW, NW><<<grid, NW * 32, S::kBytes, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_append_int2(const AppendArgs& a, int num_sms, cudaStream_t st) {
  // Few tokens (decode-time appends): one token per warp keeps the dependent
  // fmaf chains short in wall time.  Many tokens (prefill): eight tokens per
  // warp reuse each staged rotation row eight times.
  if (a.n <= 8 * num_sms / (a.Hkv > 0 ? a.Hkv : 1)) return launch_tpw<1, 8>(a, num_sms, st);
  return launch_tpw<8, 8>(a, num_sms, st);
}

cudaError_t launch_append_bf16(const AppendArgs& a, cudaStream_t st) {
  dim3 grid(a.n, a.Hkv);
  append_bf16_kernel<<<grid, 128, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq
