// fp16_cache.cu -- the FP16 paged KV cache that the quantized cache is measured
// against: prefill tokens copied into fp16 pages, and paged split-K decode
// attention over those pages on the tensor cores.
//
// The KVarN page (blog.edumints.com) states its gains relative to an FP16 KV
// cache (capacity 3-5x, throughput ~1.3x); this is that baseline, on the same
// harness.  Attention is the textbook decode of "KV Cache (Anahtar-Deger
// Onbellegi)" (yapayzekasozluk.tr), "KV Cache Nasil Calisir?" and "Paged
// Attention (vLLM)": out = softmax(scale q . k_t) v over the sequence's tokens,
// query head h reading KV head h / (Hq / Hkv).
//
// Page (per page and KV head, 65536 bytes): K then V, each [128 tokens][128
// channels] fp16.  The last page of a sequence is filled up to its length.
//
// Decode: CTA = 4 warps on one (sequence, KV head, run of pages).  The CTA
// streams half pages (64 tokens of K and of V, four 64 x 64 TMA boxes with
// 128-byte swizzle) through three stages; warp w takes tokens 16w .. 16w + 15
// of every half page with its own online-softmax state:
//   scores  S = K Q^T : mma.sync m16n8k16, A = K rows (ldmatrix), B = q (the
//           group's heads as the 8 columns, fp16, exact), fp32 accumulate;
//   values  O += V^T P : A = V^T (ldmatrix.trans), B = P (fp16 probabilities,
//           moved from the score fragments by movmatrix).
// The warps' states merge in shared memory and the splits of a (sequence, KV
// head) through the workspace, where the last CTA to arrive merges them.
#include "kvarn_internal.cuh"
#include "ptx.cuh"

namespace kvarn {
namespace {

using namespace ptx;

constexpr int kFWarps = 4;
constexpr int kFThreads = 32 * kFWarps;
constexpr int kFStages = 3;
constexpr uint32_t kFBox = 64 * 64 * 2;          // 64 tokens x 64 channels fp16
constexpr uint32_t kFStageBytes = 4 * kFBox;     // K lo, K hi, V lo, V hi
constexpr uint64_t kFWaitNs = 2000000000ull;
constexpr float kFLog2e = 1.4426950408889634f;

struct __align__(1024) FSmem {
  uint8_t st[kFStages][4][kFBox];   // 96 KB; the warps' states reuse it at the end
  uint64_t full[kFStages];
  uint64_t empty[kFStages];
  int ok[kFStages];                 // stage holds a valid page
  int ticket;
};
// warp state in the reused stage memory: [warp][head]{m, l}, then
// o[warp][head][128]
constexpr int kFStateFloats = 8 * 2 + 8 * kD;
static_assert(kFWarps * kFStateFloats * 4 <= kFStages * kFStageBytes, "state fits");

__device__ __forceinline__ float fex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t fpack2(float first, float second) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(second), "f"(first));
  return r;
}
__device__ __forceinline__ uint32_t fmovm(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
// byte offset of (row, 16-byte chunk) in a 128-byte-swizzled box of 128-byte rows
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__global__ void __launch_bounds__(kFThreads, 2)
    fp16_decode_kernel(const __grid_constant__ CUtensorMap tm, const F16DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  FSmem& S = *reinterpret_cast<FSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~static_cast<uintptr_t>(1023));
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, qi = lane & 3;
  const int g = a.g;
  const float sl2 = a.scale * kFLog2e;

  int len = a.seq_lens[b];
  if (len < 0 || len > a.max_seq || (len + kT - 1) / kT > a.max_blocks) {
    if (split == 0 && kvh == 0 && tid == 0) report(a.status, KVARN_STATUS_BAD_LENGTH);
    len = 0;
  }
  const int npages = (len + kT - 1) / kT;
  const int pps = a.pages_per_split;
  const int nsb = npages > 0 ? (npages + pps - 1) / pps : 1;
  if (split >= nsb) return;
  const int u0 = split * pps, u1 = min(npages, u0 + pps);
  // half pages of this split that hold tokens
  const int h0 = 2 * u0;
  int nst = 2 * (u1 - u0);
  if (u1 == npages && nst > 0 && (len - 1) % kT < 64) --nst;   // last half page empty

  if (tid == 0) {
    for (int s = 0; s < kFStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], kFWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  const int32_t* trow = a.block_table + (int64_t)b * a.max_blocks;
  int last_issued[kFStages] = {-1, -1, -1};   // thread 0: latest load per stage
  auto issue = [&](int i, int s) {   // half page h0 + i into stage s (thread 0)
    last_issued[s] = i;
    const int hp = h0 + i, j = hp >> 1, half = hp & 1;
    const int64_t page = trow[j];
    const bool ok = page >= 0 && page < a.num_pages;
    S.ok[s] = ok;
    if (!ok) {
      report(a.status, KVARN_STATUS_BAD_PAGE);
      mbar_arrive(&S.full[s]);
      return;
    }
    mbar_arrive_expect_tx(&S.full[s], kFStageBytes);
    const int t0 = 64 * half, p = (int)page;
    tma_load_4d(S.st[s][0], &tm, 0, t0, 2 * kvh, p, &S.full[s]);
    tma_load_4d(S.st[s][1], &tm, 64, t0, 2 * kvh, p, &S.full[s]);
    tma_load_4d(S.st[s][2], &tm, 0, t0, 2 * kvh + 1, p, &S.full[s]);
    tma_load_4d(S.st[s][3], &tm, 64, t0, 2 * kvh + 1, p, &S.full[s]);
  };
  if (tid == 0)
    for (int i = 0; i < kFStages && i < nst; ++i) issue(i, i);

  // B fragments of q: lane (r, qi) holds head r (zero beyond the group), channels
  // 16 kb + 2 qi, + 1 (bq[kb][0]) and 16 kb + 8 + 2 qi, + 1 (bq[kb][1])
  uint32_t bq[8][2];
  {
    const __half* qh = a.q + ((int64_t)b * a.hq + (int64_t)kvh * g + r) * kD;
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) {
      bq[kb][0] = r < g ? __ldg(reinterpret_cast<const uint32_t*>(qh + 16 * kb + 2 * qi)) : 0u;
      bq[kb][1] = r < g ? __ldg(reinterpret_cast<const uint32_t*>(qh + 16 * kb + 8 + 2 * qi))
                        : 0u;
    }
  }

  // state for heads 2qi + e (e = 0, 1) of this lane; o rows = channels
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  float oacc[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) oacc[mt][0] = oacc[mt][1] = oacc[mt][2] = oacc[mt][3] = 0.f;
  bool timed_out = false;

  // ldmatrix lane roles: matrix mi = lane >> 3, row lane & 7
  const int mi = lane >> 3, mrow = lane & 7;
  for (int i = 0; i < nst; ++i) {
    const int s = i % kFStages;
    const uint32_t ph = (uint32_t)((i / kFStages) & 1);
    if (!mbar_wait_warp(&S.full[s], ph, kFWaitNs)) {
      timed_out = true;
      break;
    }
    if (S.ok[s]) {
      const int tok0 = 64 * (h0 + i) + 16 * warp;   // first token of this warp's tile
      // ---- scores: rows r, r + 8 (tokens), columns 2qi, 2qi + 1 (heads) ----
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const int krow = 16 * warp + mrow + 8 * (mi & 1);
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
          const uint32_t base = smem_u32(S.st[s][kb >> 2]);
          uint32_t A[4];
          ldsm_x4(A, base + swz(krow, 2 * (kb & 3) + (mi >> 1)));
          mma_16816(d, A, bq[kb][0], bq[kb][1]);
        }
      }
      const bool in0 = tok0 + r < len, in1 = tok0 + r + 8 < len;
      float sc[4] = {in0 ? d[0] * sl2 : -INFINITY, in0 ? d[1] * sl2 : -INFINITY,
                     in1 ? d[2] * sl2 : -INFINITY, in1 ? d[3] * sl2 : -INFINITY};
      float alpha[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float mx = fmaxf(sc[e], sc[e + 2]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mn = fmaxf(m[e], mx);
        if (mn == -INFINITY) {          // nothing seen yet for this head
          alpha[e] = 1.f;
          sc[e] = sc[e + 2] = 0.f;
        } else {
          alpha[e] = fex2(m[e] - mn);
          sc[e] = fex2(sc[e] - mn);
          sc[e + 2] = fex2(sc[e + 2] - mn);
        }
        m[e] = mn;
        l[e] = fmaf(l[e], alpha[e], sc[e] + sc[e + 2]);
      }
      // ---- values: P (tokens x heads) into B fragments; A = V^T tiles ----
      const uint32_t bp0 = fmovm(fpack2(sc[0], sc[1]));   // tokens 0..7
      const uint32_t bp1 = fmovm(fpack2(sc[2], sc[3]));   // tokens 8..15
      const int vrow = 16 * warp + mrow + 8 * (mi >> 1);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const uint32_t base = smem_u32(S.st[s][2 + (mt >> 2)]);
        uint32_t A[4];
        ldmatrix_x4_trans(A, base + swz(vrow, 2 * (mt & 3) + (mi & 1)));
        oacc[mt][0] *= alpha[0];
        oacc[mt][1] *= alpha[1];
        oacc[mt][2] *= alpha[0];
        oacc[mt][3] *= alpha[1];
        mma_16816(oacc[mt], A, bp0, bp1);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[s]);
    if (tid == 0 && i + kFStages < nst) {
      if (!mbar_wait_bounded(&S.empty[s], ph, kFWaitNs)) {
        report(a.status, KVARN_STATUS_TIMEOUT);
      } else {
        issue(i + kFStages, s);
      }
    }
  }
  if (timed_out) {
    if (lane == 0) report(a.status, KVARN_STATUS_TIMEOUT);
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) oacc[mt][0] = oacc[mt][1] = oacc[mt][2] = oacc[mt][3] = 0.f;
  }
  // no copy into the stages may still be in flight when they are reused:
  // thread 0 waits (bounded) for the latest load of each stage, which every
  // consumer has normally waited for already
  if (tid == 0) {
#pragma unroll
    for (int st = 0; st < kFStages; ++st)
      if (last_issued[st] >= 0)
        mbar_wait_bounded(&S.full[st], (uint32_t)((last_issued[st] / kFStages) & 1), kFWaitNs);
  }
  __syncthreads();

  float* const sw = reinterpret_cast<float*>(&S.st[0][0][0]) + warp * kFStateFloats;
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    float ls = l[e];
    ls += __shfl_xor_sync(0xffffffffu, ls, 4);
    ls += __shfl_xor_sync(0xffffffffu, ls, 8);
    ls += __shfl_xor_sync(0xffffffffu, ls, 16);
    const int h = 2 * qi + e;
    if (r == 0) {
      sw[2 * h] = m[e];
      sw[2 * h + 1] = ls;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      sw[16 + h * kD + 16 * mt + r] = oacc[mt][e];
      sw[16 + h * kD + 16 * mt + 8 + r] = oacc[mt][2 + e];
    }
  }
  __syncthreads();

  // ---- merge the warps; the result goes to the output (one split) or to
  // this split's partial state ----
  __half* ob = a.out + ((int64_t)b * a.hq + (int64_t)kvh * g) * kD;
  const float* st0 = reinterpret_cast<const float*>(&S.st[0][0][0]);
  for (int i = tid; i < g * kD; i += kFThreads) {
    const int h = i >> 7, ch = i & 127;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kFWarps; ++w) M = fmaxf(M, st0[w * kFStateFloats + 2 * h]);
    float o = 0.f, L = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kFWarps; ++w) {
        const float* x = st0 + w * kFStateFloats;
        const float wt = fex2(x[2 * h] - M);
        o = fmaf(wt, x[16 + h * kD + ch], o);
        L = fmaf(wt, x[2 * h + 1], L);
      }
    }
    if (nsb == 1) {
      ob[i] = __float2half_rn(L > 0.f ? o / L : 0.f);
    } else {
      float* Pp =
          a.ws_part + (((int64_t)b * a.hq + kvh * g + h) * a.nsplit + split) * kPartStride;
      if (ch == 0) {
        Pp[0] = M;
        Pp[1] = L;
      }
      Pp[4 + ch] = o;
    }
  }
  if (nsb == 1) return;
  __threadfence();
  __syncthreads();
  if (tid == 0) S.ticket = atomicAdd(a.ws_count + (int64_t)b * a.hkv + kvh, 1);
  __syncthreads();
  if (S.ticket != nsb - 1) return;
  __threadfence();

  // ---- last split to arrive: merge all splits (warp w: heads w, w + 4) ----
  for (int h = warp; h < g; h += kFWarps) {
    const float* P0 = a.ws_part + (((int64_t)b * a.hq + kvh * g + h) * a.nsplit) * kPartStride;
    float M = -INFINITY, L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sp = 0; sp < nsb; ++sp) {
      const float* Ps = P0 + (int64_t)sp * kPartStride;
      const float2 ml = __ldcg(reinterpret_cast<const float2*>(Ps));
      if (ml.x == -INFINITY) continue;
      const float4 os = __ldcg(reinterpret_cast<const float4*>(Ps + 4) + lane);
      const float Mn = fmaxf(M, ml.x);
      const float al = fex2(M - Mn), wt = fex2(ml.x - Mn);
      L = fmaf(L, al, wt * ml.y);
      acc.x = fmaf(acc.x, al, wt * os.x);
      acc.y = fmaf(acc.y, al, wt * os.y);
      acc.z = fmaf(acc.z, al, wt * os.z);
      acc.w = fmaf(acc.w, al, wt * os.w);
      M = Mn;
    }
    const float il = L > 0.f ? 1.f / L : 0.f;
    __half2 o01 = __floats2half2_rn(acc.x * il, acc.y * il);
    __half2 o23 = __floats2half2_rn(acc.z * il, acc.w * il);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&o01);
    pk.y = *reinterpret_cast<uint32_t*>(&o23);
    *reinterpret_cast<uint2*>(ob + h * kD + 4 * lane) = pk;
  }
  if (tid == 0) a.ws_count[(int64_t)b * a.hkv + kvh] = 0;
}

// Tokens [128 j, min(len, 128 j + 128)) of sequence b, KV head h, into page
// block_table[b][j].  grid (ceil(max_seq / 128), hkv, batch), block 256.
__global__ void __launch_bounds__(256) fp16_write_kernel(F16WriteArgs a) {
  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int len = a.seq_lens[b];
  if (len < 0 || len > a.max_seq) {
    if (j == 0 && h == 0 && threadIdx.x == 0) report(a.status, KVARN_STATUS_BAD_LENGTH);
    return;
  }
  const int n = min(kT, len - kT * j);
  if (n <= 0) return;
  if (j >= a.max_blocks) {
    if (threadIdx.x == 0) report(a.status, KVARN_STATUS_BAD_LENGTH);
    return;
  }
  const int64_t page = a.block_table[(int64_t)b * a.max_blocks + j];
  if (page < 0 || page >= a.num_pages) {
    if (threadIdx.x == 0) report(a.status, KVARN_STATUS_BAD_PAGE);
    return;
  }
  uint8_t* dst = a.pool + (page * a.hkv + h) * (int64_t)kF16PageBytes;
  for (int part = 0; part < 2; ++part) {
    const __half* src = (part ? a.v : a.k) + (int64_t)b * a.sb + (int64_t)h * a.sh;
    uint4* d = reinterpret_cast<uint4*>(dst + part * (kT * kD * 2));
    for (int x = threadIdx.x; x < n * (kD / 8); x += blockDim.x) {
      const int t = x / (kD / 8), c = x % (kD / 8);
      d[t * (kD / 8) + c] =
          __ldg(reinterpret_cast<const uint4*>(src + (int64_t)(kT * j + t) * a.st) + c);
    }
  }
}

constexpr int kFSmemBytes = (int)sizeof(FSmem) + 1024;

}  // namespace

// Resident CTAs per SM of the decode kernel (shared memory bound).
constexpr int kF16CtasPerSm = 233472 / (kFSmemBytes + 1024);

DecodePlan fp16_decode_plan(int batch, int hq, int hkv, int max_seq, int num_sms) {
  DecodePlan p{};
  (void)hq;
  const int64_t units = max_seq > 0 ? ((int64_t)max_seq + kT - 1) / kT : 1;
  const int64_t groups = (int64_t)batch * hkv;
  const int64_t slots = (int64_t)(num_sms > 0 ? num_sms : 1) * kF16CtasPerSm;
  int64_t ns = slots / (groups > 0 ? groups : 1);
  const int64_t ns_cap = (units + 1) / 2;    // at least two pages per split
  if (ns > ns_cap) ns = ns_cap;
  if (ns < 1) ns = 1;
  const int64_t pps = (units + ns - 1) / ns;
  p.pages_per_split = (int)pps;
  p.nsplit = (int)((units + pps - 1) / pps);
  if (p.nsplit > 1) {
    p.part_bytes = (size_t)batch * hq * p.nsplit * kPartStride * sizeof(float);
    p.part_bytes = (p.part_bytes + 255) & ~(size_t)255;
    p.count_bytes = ((size_t)batch * hkv * sizeof(int) + 255) & ~(size_t)255;
  }
  return p;
}

cudaError_t launch_fp16_write(const F16WriteArgs& a, cudaStream_t s) {
  if (a.max_seq <= 0) return cudaSuccess;
  dim3 grid((a.max_seq + kT - 1) / kT, a.hkv, a.batch);
  fp16_write_kernel<<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_fp16_decode(const F16DecodeArgs& a, const void* pool, cudaStream_t s) {
  static std::atomic<uint64_t> smem_set{0};
  cudaError_t e = ensure_dynamic_smem(fp16_decode_kernel, kFSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  // pool as (channel, token, 2 * head + part, page), 64 x 64 boxes
  CUtensorMap tm;
  const uint64_t dims[4] = {(uint64_t)kD, (uint64_t)kT, (uint64_t)2 * a.hkv,
                            (uint64_t)(a.num_pages > 0 ? a.num_pages : 1)};
  const uint64_t strides[3] = {(uint64_t)kD * 2, (uint64_t)kT * kD * 2,
                               (uint64_t)a.hkv * kF16PageBytes};
  const uint32_t box[4] = {64, 64, 1, 1};
  if (!encode_fp16_map_4d(&tm, pool, dims, strides, box)) return cudaErrorInvalidValue;
  dim3 grid(a.nsplit, a.hkv, a.batch);
  fp16_decode_kernel<<<grid, kFThreads, kFSmemBytes, s>>>(tm, a);
  return cudaGetLastError();
}

}  // namespace kvarn
