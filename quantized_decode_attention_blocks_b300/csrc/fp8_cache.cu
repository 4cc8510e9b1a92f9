// fp8_cache.cu -- the FP8 paged KV cache, the second baseline the quantized
// cache is measured against: prefill tokens quantized to e4m3 with one fp32
// scale per token and KV head, and paged split-K decode attention over them.
//
// The glossary "KV Cache (Anahtar-Deger Onbellegi)" (yapayzekasozluk.tr),
// "Sik Sorulan Sorular", names INT8/FP8 quantization as the common way to
// halve the KV cache.  Readings: e4m3 (largest finite 448), s = max|x| / 448
// per token and head, codes e4m3(x / s) rounded to nearest even and saturated;
// the two divisions are fp32 (IEEE), so that the codes are the ones the
// float64 oracle decides in the same precision.
//
// Page (per page and KV head, KVARN_FP8_PAGE_BYTES = 33792 bytes):
//   [0, 16384)       K codes [128 tokens][128 channels] e4m3
//   [16384, 32768)   V codes, same
//   [32768, 33280)   K scales fp32 [128 tokens]
//   [33280, 33792)   V scales fp32 [128 tokens]
//
// Decode: the structure of the FP16 decode (fp16_cache.cu): CTA = 4 warps on
// one (sequence, KV head, run of pages), half pages (64 tokens) streamed
// through four stages by bulk copies (codes and scales: 16.5 KB), warp w on
// tokens 16w .. 16w + 15 with its own online-softmax state.  Each warp turns
// its 16 rows of codes into fp16 (exact: every e4m3 value is an fp16 value)
// in its own rows of four 64 x 64 swizzled boxes, then runs the FP16 decode's
// mma.sync fragments on them; the per-token scales multiply the fp32 scores
// and fold into the probabilities of the value sum.
#include "kvarn_internal.cuh"
#include "ptx.cuh"

namespace kvarn {
namespace {

using namespace ptx;

constexpr int kPWarps = 4;
constexpr int kPThreads = 32 * kPWarps;
constexpr int kPStages = 4;
constexpr uint32_t kPHalf = 64 * kD;             // codes of 64 tokens: 8 KB
constexpr uint32_t kPBox = 64 * 64 * 2;          // fp16 box 64 rows x 64 channels
constexpr uint32_t kPStageTx = 2 * kPHalf + 2 * 64 * 4;
constexpr uint64_t kPWaitNs = 2000000000ull;
constexpr float kPLog2e = 1.4426950408889634f;
// the value-sum probabilities carry this power of two, so that p * s^V stays
// in fp16's normal range for small scales; removed at the end
constexpr float kPVBoost = 64.f;

struct __align__(1024) PSmem {
  uint8_t kc[kPStages][kPHalf];
  uint8_t vc[kPStages][kPHalf];
  float ks[kPStages][64];
  float vs[kPStages][64];
  uint8_t box[4][kPBox];            // fp16 K lo, K hi, V lo, V hi; warp w owns rows 16w ..
  uint64_t full[kPStages];
  uint64_t empty[kPStages];
  int ok[kPStages];
  int ticket;
};
constexpr int kPStateFloats = 8 * 2 + 8 * kD;    // per warp: [head]{m, l}, o[head][128]
static_assert(kPWarps * kPStateFloats * 4 <= 2 * kPStages * kPHalf, "state fits in the codes");
constexpr int kPSmemBytes = (int)sizeof(PSmem) + 1024;

__device__ __forceinline__ float pex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t ppack2(float first, float second) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(second), "f"(first));
  return r;
}
__device__ __forceinline__ uint32_t pmovm(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}
__device__ __forceinline__ void pldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ uint32_t pswz(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}
// two e4m3 codes (first in the low byte) -> fp16x2 (first in the low half)
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t r;
  const unsigned short h = (unsigned short)(two & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(h));
  return r;
}
// two fp32 -> e4m3 codes, first in the low byte, nearest even, saturated
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float first, float second) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(second), "f"(first));
  return r;
}

__global__ void __launch_bounds__(kPThreads, 2)
    fp8_decode_kernel(const F16DecodeArgs a, const uint8_t* __restrict__ pool) {
  extern __shared__ uint8_t smem_raw[];
  PSmem& S = *reinterpret_cast<PSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~static_cast<uintptr_t>(1023));
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, qi = lane & 3;
  const int g = a.g;
  const float sl2 = a.scale * kPLog2e;

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
  const int h0 = 2 * u0;
  int nst = 2 * (u1 - u0);
  if (u1 == npages && nst > 0 && (len - 1) % kT < 64) --nst;   // last half page empty

  if (tid == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], kPWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  const int32_t* trow = a.block_table + (int64_t)b * a.max_blocks;
  int last_issued[kPStages] = {-1, -1, -1, -1};   // thread 0: latest load per stage
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
    const uint8_t* pg = pool + (page * a.hkv + kvh) * (int64_t)KVARN_FP8_PAGE_BYTES;
    mbar_arrive_expect_tx(&S.full[s], kPStageTx);
    bulk_g2s(S.kc[s], pg + kPHalf * half, kPHalf, &S.full[s]);
    bulk_g2s(S.vc[s], pg + 16384 + kPHalf * half, kPHalf, &S.full[s]);
    bulk_g2s(S.ks[s], pg + 32768 + 256 * half, 256, &S.full[s]);
    bulk_g2s(S.vs[s], pg + 33280 + 256 * half, 256, &S.full[s]);
  };
  if (tid == 0)
    for (int i = 0; i < kPStages && i < nst; ++i) issue(i, i);

  // B fragments of q (head r of the group, zero beyond it), as in the FP16 decode
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

  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  float oacc[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) oacc[mt][0] = oacc[mt][1] = oacc[mt][2] = oacc[mt][3] = 0.f;
  bool timed_out = false;

  const int mi = lane >> 3, mrow = lane & 7;
  // conversion roles: lane -> channel chunk cc (8 channels), row parity rr
  const int cc = lane & 15, rr = lane >> 4;
  for (int i = 0; i < nst; ++i) {
    const int s = i % kPStages;
    const uint32_t ph = (uint32_t)((i / kPStages) & 1);
    if (!mbar_wait_warp(&S.full[s], ph, kPWaitNs)) {
      timed_out = true;
      break;
    }
    const bool ok = S.ok[s];
    float skA = 0.f, skB = 0.f, svA = 0.f, svB = 0.f;
    if (ok) {
      // ---- this warp's 16 rows of codes -> fp16 boxes; its scales ----
#pragma unroll
      for (int it = 0; it < 8; ++it) {
        const int row = 16 * warp + 2 * it + rr;
        const uint2 k8 = *reinterpret_cast<const uint2*>(S.kc[s] + row * kD + 8 * cc);
        const uint2 v8 = *reinterpret_cast<const uint2*>(S.vc[s] + row * kD + 8 * cc);
        const uint4 kh = make_uint4(e4m3x2_to_f16x2(k8.x), e4m3x2_to_f16x2(k8.x >> 16),
                                    e4m3x2_to_f16x2(k8.y), e4m3x2_to_f16x2(k8.y >> 16));
        const uint4 vh = make_uint4(e4m3x2_to_f16x2(v8.x), e4m3x2_to_f16x2(v8.x >> 16),
                                    e4m3x2_to_f16x2(v8.y), e4m3x2_to_f16x2(v8.y >> 16));
        *reinterpret_cast<uint4*>(S.box[cc >> 3] + pswz(row, cc & 7)) = kh;
        *reinterpret_cast<uint4*>(S.box[2 + (cc >> 3)] + pswz(row, cc & 7)) = vh;
      }
      skA = S.ks[s][16 * warp + r];
      skB = S.ks[s][16 * warp + r + 8];
      svA = S.vs[s][16 * warp + r] * kPVBoost;
      svB = S.vs[s][16 * warp + r + 8] * kPVBoost;
    }
    // the stage's codes and scales are read: release it to the loader
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[s]);
    if (tid == 0 && i + kPStages < nst) {
      if (!mbar_wait_bounded(&S.empty[s], ph, kPWaitNs)) {
        report(a.status, KVARN_STATUS_TIMEOUT);
      } else {
        issue(i + kPStages, s);
      }
    }
    __syncwarp();   // warp 0 reconverges after its loader thread's wait
    if (ok) {
      const int tok0 = 64 * (h0 + i) + 16 * warp;
      // ---- scores: rows r, r + 8 (tokens), columns 2qi, 2qi + 1 (heads) ----
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      {
        const int krow = 16 * warp + mrow + 8 * (mi & 1);
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
          uint32_t A[4];
          pldsm_x4(A, smem_u32(S.box[kb >> 2]) + pswz(krow, 2 * (kb & 3) + (mi >> 1)));
          mma_16816(d, A, bq[kb][0], bq[kb][1]);
        }
      }
      const bool in0 = tok0 + r < len, in1 = tok0 + r + 8 < len;
      float sc[4] = {in0 ? d[0] * skA * sl2 : -INFINITY, in0 ? d[1] * skA * sl2 : -INFINITY,
                     in1 ? d[2] * skB * sl2 : -INFINITY, in1 ? d[3] * skB * sl2 : -INFINITY};
      float alpha[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float mx = fmaxf(sc[e], sc[e + 2]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mn = fmaxf(m[e], mx);
        if (mn == -INFINITY) {
          alpha[e] = 1.f;
          sc[e] = sc[e + 2] = 0.f;
        } else {
          alpha[e] = pex2(m[e] - mn);
          sc[e] = pex2(sc[e] - mn);
          sc[e + 2] = pex2(sc[e + 2] - mn);
        }
        m[e] = mn;
        l[e] = fmaf(l[e], alpha[e], sc[e] + sc[e + 2]);
      }
      // ---- values: p s^V (boosted) into B fragments; A = V^T tiles ----
      const uint32_t bp0 = pmovm(ppack2(sc[0] * svA, sc[1] * svA));   // tokens 0..7
      const uint32_t bp1 = pmovm(ppack2(sc[2] * svB, sc[3] * svB));   // tokens 8..15
      const int vrow = 16 * warp + mrow + 8 * (mi >> 1);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        uint32_t A[4];
        ldmatrix_x4_trans(A, smem_u32(S.box[2 + (mt >> 2)]) + pswz(vrow, 2 * (mt & 3) + (mi & 1)));
        oacc[mt][0] *= alpha[0];
        oacc[mt][1] *= alpha[1];
        oacc[mt][2] *= alpha[0];
        oacc[mt][3] *= alpha[1];
        mma_16816(oacc[mt], A, bp0, bp1);
      }
    }
    __syncwarp();   // this warp's boxes are read before its next conversion
  }
  if (timed_out) {
    if (lane == 0) report(a.status, KVARN_STATUS_TIMEOUT);
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) oacc[mt][0] = oacc[mt][1] = oacc[mt][2] = oacc[mt][3] = 0.f;
  }
  // no copy into the stages may still be in flight when they are reused
  if (tid == 0) {
#pragma unroll
    for (int st = 0; st < kPStages; ++st)
      if (last_issued[st] >= 0)
        mbar_wait_bounded(&S.full[st], (uint32_t)((last_issued[st] / kPStages) & 1), kPWaitNs);
  }
  __syncthreads();

  float* const sw = reinterpret_cast<float*>(&S.kc[0][0]) + warp * kPStateFloats;
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    float ls = l[e];
    ls += __shfl_xor_sync(0xffffffffu, ls, 4);
    ls += __shfl_xor_sync(0xffffffffu, ls, 8);
    ls += __shfl_xor_sync(0xffffffffu, ls, 16);
    const int h = 2 * qi + e;
    if (r == 0) {
      sw[2 * h] = m[e];
      sw[2 * h + 1] = ls * kPVBoost;   // o carries the boost
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      sw[16 + h * kD + 16 * mt + r] = oacc[mt][e];
      sw[16 + h * kD + 16 * mt + 8 + r] = oacc[mt][2 + e];
    }
  }
  __syncthreads();

  // ---- merge the warps; to the output (one split) or this split's partial ----
  __half* ob = a.out + ((int64_t)b * a.hq + (int64_t)kvh * g) * kD;
  const float* st0 = reinterpret_cast<const float*>(&S.kc[0][0]);
  for (int i = tid; i < g * kD; i += kPThreads) {
    const int h = i >> 7, ch = i & 127;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kPWarps; ++w) M = fmaxf(M, st0[w * kPStateFloats + 2 * h]);
    float o = 0.f, L = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kPWarps; ++w) {
        const float* x = st0 + w * kPStateFloats;
        const float wt = pex2(x[2 * h] - M);
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

  for (int h = warp; h < g; h += kPWarps) {
    const float* P0 = a.ws_part + (((int64_t)b * a.hq + kvh * g + h) * a.nsplit) * kPartStride;
    float M = -INFINITY, L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sp = 0; sp < nsb; ++sp) {
      const float* Ps = P0 + (int64_t)sp * kPartStride;
      const float2 ml = __ldcg(reinterpret_cast<const float2*>(Ps));
      if (ml.x == -INFINITY) continue;
      const float4 os = __ldcg(reinterpret_cast<const float4*>(Ps + 4) + lane);
      const float Mn = fmaxf(M, ml.x);
      const float al = pex2(M - Mn), wt = pex2(ml.x - Mn);
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

// Tokens [128 j, min(len, 128 j + 128)) of sequence b, KV head h, quantized
// into page block_table[b][j]: warp w takes tokens w, w + 4, ...; lane holds
// channels 4 lane .. 4 lane + 3.  grid (ceil(max_seq / 128), hkv, batch).
__global__ void __launch_bounds__(128) fp8_write_kernel(F16WriteArgs a) {
  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
  uint8_t* pg = a.pool + (page * a.hkv + h) * (int64_t)KVARN_FP8_PAGE_BYTES;
  for (int part = 0; part < 2; ++part) {
    const __half* src = (part ? a.v : a.k) + (int64_t)b * a.sb + (int64_t)h * a.sh;
    uint8_t* codes = pg + part * 16384;
    float* scales = reinterpret_cast<float*>(pg + 32768 + part * 512);
    for (int t = warp; t < n; t += 4) {
      const uint2 raw =
          __ldg(reinterpret_cast<const uint2*>(src + (int64_t)(kT * j + t) * a.st) + lane);
      const float2 x01 = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
      const float2 x23 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
      float amax = fmaxf(fmaxf(fabsf(x01.x), fabsf(x01.y)), fmaxf(fabsf(x23.x), fabsf(x23.y)));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const float s = __fdiv_rn(amax, 448.f);
      uint32_t w = 0u;
      if (s > 0.f) {
        w = f32x2_to_e4m3x2(__fdiv_rn(x01.x, s), __fdiv_rn(x01.y, s)) |
            (f32x2_to_e4m3x2(__fdiv_rn(x23.x, s), __fdiv_rn(x23.y, s)) << 16);
      }
      reinterpret_cast<uint32_t*>(codes + t * kD)[lane] = w;
      if (lane == 0) scales[t] = s;
    }
  }
}

}  // namespace

// Resident CTAs per SM of the FP8 decode kernel (shared memory bound).
constexpr int kFp8CtasPerSm = 233472 / (kPSmemBytes + 1024);

DecodePlan fp8_decode_plan(int batch, int hq, int hkv, int max_seq, int num_sms) {
  DecodePlan p{};
  const int64_t units = max_seq > 0 ? ((int64_t)max_seq + kT - 1) / kT : 1;
  const int64_t groups = (int64_t)batch * hkv;
  const int64_t slots = (int64_t)(num_sms > 0 ? num_sms : 1) * kFp8CtasPerSm;
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

cudaError_t launch_fp8_write(const F16WriteArgs& a, cudaStream_t s) {
  if (a.max_seq <= 0) return cudaSuccess;
  dim3 grid((a.max_seq + kT - 1) / kT, a.hkv, a.batch);
  fp8_write_kernel<<<grid, 128, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_fp8_decode(const F16DecodeArgs& a, const void* pool, cudaStream_t s) {
  static std::atomic<uint64_t> smem_set{0};
  cudaError_t e = ensure_dynamic_smem(fp8_decode_kernel, kPSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  dim3 grid(a.nsplit, a.hkv, a.batch);
  fp8_decode_kernel<<<grid, kPThreads, kPSmemBytes, s>>>(a, static_cast<const uint8_t*>(pool));
  return cudaGetLastError();
}

}  // namespace kvarn
