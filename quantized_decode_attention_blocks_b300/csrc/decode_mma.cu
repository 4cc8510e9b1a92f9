// decode_mma.cu -- paged split-K decode attention over the quantized cache on
// the tensor cores (mma.sync m16n8k16, fp16 x fp16 -> fp32).
//
// Method: one new query token per sequence attends to every cached token
// ("KV Cache (Anahtar-Deger Onbellegi)", yapayzekasozluk.tr, "KV Cache Nasil
// Calisir?"), several query heads sharing one KV head ("Sik Sorulan
// Sorular", GQA).  Keys and values are stored rotated (y = H x, the KVarN
// page, blog.edumints.com, "KVarN Nasil Calisir?", stage "Dondurulmus
// Onbellek": the orthonormal rotation keeps attention scores), so:
//   score_t = q~ . yhat_t,   q~ = H q,   yhat_td = c_d (s'_t q_td + z'_t)
//           = s'_t * sum_d (q~_d c_d) q_td + z'_t * sum_d q~_d c_d
//   o = H (sum_t p_t yhatV_t) + sum_tail p_t v_t,
//   sum_t p_t yhatV_td = cV_d (sum_t (p_t s'V_t) qV_td + sum_t p_t z'V_t).
// The two inner sums over codes are dense contractions of a 128x128 page of
// small integers (exact in fp16) with a query-side factor; they run as
// mma.sync with the codes unpacked straight into A fragments by bit tricks
// (1024 + q is an exact fp16; subtracting 1024 leaves q).  The query-side
// factor is split into an fp16 pair hi + lo (and scaled by a power of two to
// stay in fp16 range), giving ~22 significant bits with fp32 accumulation.
//
// One CTA = one warp = one (sequence, KV head, split of pages); the g query
// heads of the group share every page it reads.  Each warp streams its pages
// through a private double buffer: cp.async.bulk (TMA engine) copies the
// 15360-byte record of (page, KV head) into shared memory, completing on an
// mbarrier, while the warp computes on the other buffer.  Every wait is
// bounded; on expiry the CTA reports KVARN_STATUS_TIMEOUT and drains.
// The split owning the end of the sequence also adds the fp16 tail.  Partial
// softmax states of the splits are merged (log-sum-exp) by the last CTA of
// each (sequence, KV head) to arrive, in the same launch.
#include "kvarn_internal.cuh"
#include "ptx.cuh"

namespace kvarn {
namespace {

using namespace ptx;

constexpr uint32_t kMagic = 0x64006400u;       // fp16x2 (1024, 1024)
constexpr uint32_t kH16 = 0x2C002C00u;         // fp16x2 (1/16, 1/16)
constexpr uint32_t kNeg64 = 0xD400D400u;       // fp16x2 (-64, -64)
constexpr uint32_t kQuarter = 0x34003400u;     // fp16x2 (1/4, 1/4)
constexpr uint32_t kNeg256 = 0xDC00DC00u;      // fp16x2 (-256, -256)
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;

template <int NT>
struct __align__(128) MmaSmem {
  uint8_t kst[kKPart];           // K part of the current page record
  uint8_t vst[kVPart];           // V part of the current page record
  float qrot[4 * NT][kD];        // H q per (padded) head
  uint32_t pbuf[kT * 4 * NT];    // P' hi/lo, [token][n-tile][4 x f16x2]
  uint64_t bar[2];               // 0: K part landed, 1: V part landed
  float mh[4 * NT], lh[4 * NT];
};

// nibble pairs of a 32-bit word: (n_j, n_{j+4}) as an fp16x2
__device__ __forceinline__ uint32_t nib_lo(uint32_t w) {   // j = 0 (or 2 after >> 8)
  return hsub2_u32(lop_and_or(w, 0x000F000Fu, kMagic), kMagic);
}
__device__ __forceinline__ uint32_t nib_hi(uint32_t w) {   // j = 1 (or 3 after >> 8)
  return hfma2_u32(lop_and_or(w, 0x00F000F0u, kMagic), kH16, kNeg64);
}
// crumb pairs of a 32-bit word shifted right by 4i: (c_{2i}, c_{2i+8}) and (c_{2i+1}, c_{2i+9})
__device__ __forceinline__ uint32_t crumb_a(uint32_t x) {
  return hsub2_u32(lop_and_or(x, 0x00030003u, kMagic), kMagic);
}
__device__ __forceinline__ uint32_t crumb_b(uint32_t x) {
  return hfma2_u32(lop_and_or(x, 0x000C000Cu, kMagic), kQuarter, kNeg256);
}

// 2^k scale that maps amax into [2^14, 2^15), and its inverse.
__device__ __forceinline__ void pow2_scale(float amax, float& s, float& inv) {
  const int e = (__float_as_int(amax) >> 23) & 0xff;
  const int se = min(max(268 - e, 1), 253);
  s = __int_as_float(se << 23);
  inv = __int_as_float((254 - se) << 23);
}

// Veltkamp split of x into an 11-bit head (exact in fp16 when in range) and a
// tail.  The _rn intrinsics keep the compiler from contracting c - x into an
// FMA, which would return x itself as the head.
__device__ __forceinline__ void split11(float x, float& hi, float& lo) {
  const float c = __fmul_rn(x, 8193.0f);   // 2^13 + 1: 24 - 13 = 11 head bits
  hi = __fsub_rn(c, __fsub_rn(c, x));
  lo = __fsub_rn(x, hi);
}

__device__ __forceinline__ float warp_max_r(float x) {   // over lanes sharing lane & 3
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 4));
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 8));
  return fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 16));
}
__device__ __forceinline__ float warp_sum_r(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 4);
  x += __shfl_xor_sync(0xffffffffu, x, 8);
  return x + __shfl_xor_sync(0xffffffffu, x, 16);
}

// In-place scaled Walsh-Hadamard transform of n rows of 128 floats, one warp.
__device__ __forceinline__ void warp_fwht(float (*v)[kD], int n) {
  const int lane = threadIdx.x;
  for (int s = 1; s < kD; s <<= 1) {
    for (int i = lane; i < n * (kD / 2); i += 32) {
      const int h = i >> 6, k = i & 63;
      const int lo = ((k & ~(s - 1)) << 1) | (k & (s - 1));
      const float x = v[h][lo], y = v[h][lo + s];
      v[h][lo] = x + y;
      v[h][lo + s] = x - y;
    }
    __syncwarp();
  }
  for (int i = lane; i < n * kD; i += 32) v[i >> 7][i & 127] *= kInvSqrt128;
  __syncwarp();
}

template <int NT>
__global__ void __launch_bounds__(32) decode_mma_kernel(DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  MmaSmem<NT>& S = *reinterpret_cast<MmaSmem<NT>*>(smem_raw);
  constexpr int G = 4 * NT;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int lane = threadIdx.x, r = lane >> 2, qi = lane & 3;
  const int g = a.g;
  const float sl2 = a.scale * kLog2e;   // scores are kept in log2 units

  int len = a.seq_lens[b];
  if (len < 0 || len > a.max_seq || len / kT > a.max_blocks) {
    if (split == 0 && kvh == 0 && lane == 0) report(a.status, KVARN_STATUS_BAD_LENGTH);
    len = 0;
  }
  const int nfull = len / kT, rem = len % kT;
  const int pps = a.pages_per_split;
  const int nsb = nfull > 0 ? (nfull + pps - 1) / pps : 1;
  if (split >= nsb) return;
  const int u0 = split * pps, u1 = min(nfull, u0 + pps);
  const bool has_tail = split == nsb - 1 && rem > 0;

  if (lane == 0) {
    mbar_init(&S.bar[0], 1);
    mbar_init(&S.bar[1], 1);
    fence_mbar_init();
  }
  __syncwarp();

  const int32_t* trow = a.block_table + (int64_t)b * a.max_blocks;
  auto page_of = [&](int u) -> int64_t {
    if (u >= u1) return -1;
    const int64_t p = trow[u];
    if (p < 0 || p >= a.num_pages) {
      if (lane == 0) report(a.status, KVARN_STATUS_BAD_PAGE);
      return -1;
    }
    return p;
  };
  auto rec_of = [&](int64_t page) { return a.pool + (page * a.hkv + kvh) * (int64_t)kRec; };
  auto issue_k = [&](int64_t page) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&S.bar[0], kKPart);
      bulk_g2s(S.kst, rec_of(page), kKPart, &S.bar[0]);
    }
  };
  auto issue_v = [&](int64_t page) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&S.bar[1], kVPart);
      bulk_g2s(S.vst, rec_of(page) + kKPart, kVPart, &S.bar[1]);
    }
  };

  // first page in flight while the query is rotated
  int64_t cur = page_of(u0);
  bool k_busy = false, v_busy = false;
  uint32_t kph = 0, vph = 0;
  if (cur >= 0) {
    issue_k(cur);
    issue_v(cur);
    k_busy = v_busy = true;
  }
  {
    const __half* qb = a.q + ((int64_t)b * a.hq + (int64_t)kvh * g) * kD;
    for (int i = lane; i < G * kD; i += 32) {
      const int h = i >> 7;
      S.qrot[h][i & 127] = h < g ? __half2float(qb[i]) : 0.f;
    }
    __syncwarp();
    warp_fwht(S.qrot, G);
  }

  float m[NT], l[NT], oacc[NT][16];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m[nt] = -INFINITY;
    l[nt] = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) oacc[nt][j] = 0.f;
  }
  bool timed_out = false;

  for (int u = u0; u < u1; ++u) {
    float sc[NT][16];
    if (cur >= 0) {
      if (!mbar_wait_bounded(&S.bar[0], kph, kWaitLimitNs)) {
        timed_out = true;
        break;
      }
      kph ^= 1;
      k_busy = false;
      const uint8_t* P = S.kst;

      // ---- query-side B fragments: qc = q~ * cK, scaled, split hi / lo ----
      uint32_t bq[NT][8][2];
      float sumq[NT], invq[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int h = 4 * nt + (r >> 1);
        const float4* qv = reinterpret_cast<const float4*>(&S.qrot[h][32 * qi]);
        const float4* cv = reinterpret_cast<const float4*>(P + kOffKC + 128 * qi);
        float v[32];
        float amax = 0.f, sum = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float4 q4 = qv[k], c4 = cv[k];
          v[4 * k + 0] = q4.x * c4.x;
          v[4 * k + 1] = q4.y * c4.y;
          v[4 * k + 2] = q4.z * c4.z;
          v[4 * k + 3] = q4.w * c4.w;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            amax = fmaxf(amax, fabsf(v[4 * k + e]));
            sum += v[4 * k + e];
          }
        }
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        float scl, inv;
        pow2_scale(amax, scl, inv);
        const bool lo_part = r & 1;
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
#pragma unroll
          for (int slot = 0; slot < 2; ++slot) {
            const int c0 = 8 * (kb >> 1) + 2 * (kb & 1) + slot;
            float h0, l0, h1, l1;
            split11(v[c0] * scl, h0, l0);
            split11(v[c0 + 4] * scl, h1, l1);
            bq[nt][kb][slot] = lo_part ? pack_f16x2(l0, l1) : pack_f16x2(h0, h1);
          }
        }
        // this lane's score head is 4nt + qi: fetch its sum and scale
        sumq[nt] = __shfl_sync(0xffffffffu, sum, 8 * qi);
        invq[nt] = __shfl_sync(0xffffffffu, inv, 8 * qi);
      }

      // ---- scores: K codes (A) x qc (B) ----
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const int tA = 16 * mt + r, tB = tA + 8;
        const uint4 wa = *reinterpret_cast<const uint4*>(P + kOffKCodes + 64 * tA + 16 * qi);
        const uint4 wb = *reinterpret_cast<const uint4*>(P + kOffKCodes + 64 * tB + 16 * qi);
        const uint32_t WA[4] = {wa.x, wa.y, wa.z, wa.w};
        const uint32_t WB[4] = {wb.x, wb.y, wb.z, wb.w};
        float d[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
#pragma unroll
        for (int mw = 0; mw < 4; ++mw) {
          {
            const uint32_t A[4] = {nib_lo(WA[mw]), nib_lo(WB[mw]), nib_hi(WA[mw]),
                                   nib_hi(WB[mw])};
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma_16816(d[nt], A, bq[nt][2 * mw][0], bq[nt][2 * mw][1]);
          }
          {
            const uint32_t xa = WA[mw] >> 8, xb = WB[mw] >> 8;
            const uint32_t A[4] = {nib_lo(xa), nib_lo(xb), nib_hi(xa), nib_hi(xb)};
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma_16816(d[nt], A, bq[nt][2 * mw + 1][0], bq[nt][2 * mw + 1][1]);
          }
        }
        const float2 szA = *reinterpret_cast<const float2*>(P + kOffKSZ + 8 * tA);
        const float2 szB = *reinterpret_cast<const float2*>(P + kOffKSZ + 8 * tB);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float dA = (d[nt][0] + d[nt][1]) * invq[nt];
          const float dB = (d[nt][2] + d[nt][3]) * invq[nt];
          sc[nt][2 * mt] = sl2 * fmaf(szA.x, dA, szA.y * sumq[nt]);
          sc[nt][2 * mt + 1] = sl2 * fmaf(szB.x, dB, szB.y * sumq[nt]);
        }
      }
    }
    __syncwarp();   // the K part of this page is consumed
    const int64_t nxt = page_of(u + 1);
    if (nxt >= 0) {
      issue_k(nxt);
      k_busy = true;
    }
    if (cur >= 0) {
      // ---- online softmax (log2 units) ----
      float alpha[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float pm = sc[nt][0];
#pragma unroll
        for (int j = 1; j < 16; ++j) pm = fmaxf(pm, sc[nt][j]);
        pm = warp_max_r(pm);
        const float mnew = fmaxf(m[nt], pm);
        alpha[nt] = m[nt] == -INFINITY ? 0.f : exp2f(m[nt] - mnew);
        m[nt] = mnew;
        float ls = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          sc[nt][j] = exp2f(sc[nt][j] - mnew);   // now p
          ls += sc[nt][j];
        }
        l[nt] = fmaf(l[nt], alpha[nt], ls);
      }

      if (!mbar_wait_bounded(&S.bar[1], vph, kWaitLimitNs)) {
        timed_out = true;
        break;
      }
      vph ^= 1;
      v_busy = false;

      // ---- P' = p * s'V (scaled, hi/lo) into shared memory; z' sums ----
      float smax = 0.f;
      float2 szv[16];
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        szv[2 * mt] = *reinterpret_cast<const float2*>(S.vst + (kOffVSZ - kKPart) + 8 * (16 * mt + r));
        szv[2 * mt + 1] = *reinterpret_cast<const float2*>(S.vst + (kOffVSZ - kKPart) + 8 * (16 * mt + r + 8));
        smax = fmaxf(smax, fmaxf(fabsf(szv[2 * mt].x), fabsf(szv[2 * mt + 1].x)));
      }
      smax = warp_max_r(smax);
      float fs, finv;
      pow2_scale(smax, fs, finv);
      float zpage[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float zp = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int tok = 16 * (j >> 1) + r + 8 * (j & 1);
          float hi, lo;
          split11(sc[nt][j] * szv[j].x * fs, hi, lo);
          S.pbuf[tok * 4 * NT + nt * 4 + qi] = pack_f16x2(hi, lo);
          zp = fmaf(sc[nt][j], szv[j].y, zp);
        }
        zpage[nt] = warp_sum_r(zp);
      }
      __syncwarp();

      // ---- value sum: V codes (A) x P' (B) ----
      uint32_t bp[NT][8][2];
      {
        const int mu = lane >> 3, rho = lane & 7;
        const int slot = mu & 1;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int kb0 = 0; kb0 < 8; kb0 += 2) {
            const int kbm = kb0 + (mu >> 1);
            const int tok = 16 * kbm + 2 * (rho >> 1) + slot + 8 * (rho & 1);
            uint32_t rr[4];
            ldmatrix_x4_trans(rr, smem_u32(&S.pbuf[tok * 4 * NT + nt * 4]));
            bp[nt][kb0][0] = rr[0];
            bp[nt][kb0][1] = rr[1];
            bp[nt][kb0 + 1][0] = rr[2];
            bp[nt][kb0 + 1][1] = rr[3];
          }
        }
      }
      const float* cvv = reinterpret_cast<const float*>(S.vst + (kOffVC - kKPart));
#pragma unroll
      for (int mc = 0; mc < 8; ++mc) {
        const int cA = 16 * mc + r, cB = cA + 8;
        const uint4 a0 = *reinterpret_cast<const uint4*>(S.vst + (kOffVCodes - kKPart) + 32 * cA);
        const uint4 a1 = *reinterpret_cast<const uint4*>(S.vst + (kOffVCodes - kKPart) + 32 * cA + 16);
        const uint4 b0 = *reinterpret_cast<const uint4*>(S.vst + (kOffVCodes - kKPart) + 32 * cB);
        const uint4 b1 = *reinterpret_cast<const uint4*>(S.vst + (kOffVCodes - kKPart) + 32 * cB + 16);
        const uint32_t WA[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const uint32_t WB[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        float d[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
#pragma unroll
        for (int kb = 0; kb < 8; ++kb) {
          const uint32_t xa = WA[kb] >> (4 * qi), xb = WB[kb] >> (4 * qi);
          const uint32_t A[4] = {crumb_a(xa), crumb_a(xb), crumb_b(xa), crumb_b(xb)};
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_16816(d[nt], A, bp[nt][kb][0], bp[nt][kb][1]);
        }
        const float cvA = cvv[cA], cvB = cvv[cB];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          oacc[nt][2 * mc] =
              fmaf(oacc[nt][2 * mc], alpha[nt], cvA * fmaf(d[nt][0] + d[nt][1], finv, zpage[nt]));
          oacc[nt][2 * mc + 1] = fmaf(oacc[nt][2 * mc + 1], alpha[nt],
                                      cvB * fmaf(d[nt][2] + d[nt][3], finv, zpage[nt]));
        }
      }
    }
    __syncwarp();   // the V part (and pbuf) of this page is consumed
    if (nxt >= 0) {
      issue_v(nxt);
      v_busy = true;
    }
    cur = nxt;
  }

  if (timed_out) {
    report(a.status, KVARN_STATUS_TIMEOUT);
    // drain copies still in flight before the CTA's shared memory is released
    if (k_busy) mbar_wait_bounded(&S.bar[0], kph, kWaitLimitNs);
    if (v_busy) mbar_wait_bounded(&S.bar[1], vph, kWaitLimitNs);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) m[nt] = -INFINITY, l[nt] = 0.f;
  }

  // ---- flatten: rotated accumulator to shared memory, per-head m and l ----
  float (*O)[kD] = reinterpret_cast<float (*)[kD]>(S.kst);              // G x 128 floats
  float (*ptail)[kT] = reinterpret_cast<float (*)[kT]>(S.kst + G * kD * 4);  // G x 128
  float (*qraw)[kD] = reinterpret_cast<float (*)[kD]>(S.pbuf);          // G x 128
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const float lsum = warp_sum_r(l[nt]);
#pragma unroll
    for (int mc = 0; mc < 8; ++mc) {
      O[4 * nt + qi][16 * mc + r] = timed_out ? 0.f : oacc[nt][2 * mc];
      O[4 * nt + qi][16 * mc + r + 8] = timed_out ? 0.f : oacc[nt][2 * mc + 1];
    }
    if (r == 0) {
      S.mh[4 * nt + qi] = m[nt];
      S.lh[4 * nt + qi] = lsum;
    }
  }
  __syncwarp();
  warp_fwht(O, G);   // back to plain space

  // ---- fp16 tail (plain space): lanes over tokens for scores, channels for V ----
  float otail[G][4];
#pragma unroll
  for (int h = 0; h < G; ++h) otail[h][0] = otail[h][1] = otail[h][2] = otail[h][3] = 0.f;
  if (has_tail && !timed_out) {
    const __half* qb = a.q + ((int64_t)b * a.hq + (int64_t)kvh * g) * kD;
    for (int i = lane; i < G * kD; i += 32) {
      const int h = i >> 7;
      qraw[h][i & 127] = h < g ? __half2float(qb[i]) : 0.f;
    }
    __syncwarp();
    const __half* tkb = a.tail_k + ((int64_t)b * a.hkv + kvh) * kT * kD;
    const __half* tvb = a.tail_v + ((int64_t)b * a.hkv + kvh) * kT * kD;
    float ts[4][G];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int t = lane + 32 * j;
#pragma unroll
      for (int h = 0; h < G; ++h) ts[j][h] = -INFINITY;
      if (t < rem) {
#pragma unroll
        for (int h = 0; h < G; ++h) ts[j][h] = 0.f;
        const uint4* kr = reinterpret_cast<const uint4*>(tkb + (int64_t)t * kD);
        for (int c = 0; c < kD / 8; ++c) {
          const uint4 u = __ldg(kr + c);
          const __half2* h2 = reinterpret_cast<const __half2*>(&u);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 kf = __half22float2(h2[e]);
#pragma unroll
            for (int h = 0; h < G; ++h) {
              ts[j][h] = fmaf(qraw[h][8 * c + 2 * e], kf.x, ts[j][h]);
              ts[j][h] = fmaf(qraw[h][8 * c + 2 * e + 1], kf.y, ts[j][h]);
            }
          }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) ts[j][h] *= sl2;
      }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float tm = fmaxf(fmaxf(ts[0][h], ts[1][h]), fmaxf(ts[2][h], ts[3][h]));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, o));
      const float mold = S.mh[h];
      const float mnew = fmaxf(mold, tm);
      const float al = mold == -INFINITY ? 0.f : exp2f(mold - mnew);
      float ls = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        ts[j][h] = ts[j][h] == -INFINITY ? 0.f : exp2f(ts[j][h] - mnew);
        ls += ts[j][h];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
      __syncwarp();
      if (lane == 0) {
        S.mh[h] = mnew;
        S.lh[h] = fmaf(S.lh[h], al, ls);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) O[h][4 * lane + e] *= al;
    }
    // value sum of the tail: p through shared memory, lane owns channels 4*lane..+3
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int j = 0; j < 4; ++j) ptail[h][lane + 32 * j] = ts[j][h];
    __syncwarp();
    for (int t = 0; t < rem; ++t) {
      const uint2 vv = __ldg(reinterpret_cast<const uint2*>(tvb + (int64_t)t * kD + 4 * lane));
      const float2 v01 = __half22float2(*reinterpret_cast<const __half2*>(&vv.x));
      const float2 v23 = __half22float2(*reinterpret_cast<const __half2*>(&vv.y));
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float p = ptail[h][t];
        otail[h][0] = fmaf(p, v01.x, otail[h][0]);
        otail[h][1] = fmaf(p, v01.y, otail[h][1]);
        otail[h][2] = fmaf(p, v23.x, otail[h][2]);
        otail[h][3] = fmaf(p, v23.y, otail[h][3]);
      }
    }
  }
  __syncwarp();

  // ---- output: direct, or partial state + last-arriving merge ----
  __half* ob = a.out + ((int64_t)b * a.hq + (int64_t)kvh * g) * kD;
  if (nsb == 1) {
    for (int h = 0; h < g; ++h) {
      const float lh = S.lh[h];
      const float il = lh > 0.f ? 1.f / lh : 0.f;
      __half2 o01 = __floats2half2_rn((O[h][4 * lane] + otail[h][0]) * il,
                                      (O[h][4 * lane + 1] + otail[h][1]) * il);
      __half2 o23 = __floats2half2_rn((O[h][4 * lane + 2] + otail[h][2]) * il,
                                      (O[h][4 * lane + 3] + otail[h][3]) * il);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&o01);
      pk.y = *reinterpret_cast<uint32_t*>(&o23);
      *reinterpret_cast<uint2*>(ob + h * kD + 4 * lane) = pk;
    }
    return;
  }
  constexpr int kStride = 2 + kD;
  for (int h = 0; h < g; ++h) {
    float* Pp = a.ws_part + (((int64_t)b * a.hq + kvh * g + h) * a.nsplit + split) * kStride;
    if (lane == 0) {
      Pp[0] = S.mh[h];
      Pp[1] = S.lh[h];
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) Pp[2 + 4 * lane + e] = O[h][4 * lane + e] + otail[h][e];
  }
  __threadfence();
  __syncwarp();
  int ticket = 0;
  if (lane == 0) ticket = atomicAdd(a.ws_count + (int64_t)b * a.hkv + kvh, 1);
  ticket = __shfl_sync(0xffffffffu, ticket, 0);
  if (ticket != nsb - 1) return;
  __threadfence();
  for (int h = 0; h < g; ++h) {
    const float* Pp = a.ws_part + (((int64_t)b * a.hq + kvh * g + h) * a.nsplit) * kStride;
    float M = -INFINITY;
    for (int s2 = lane; s2 < nsb; s2 += 32) M = fmaxf(M, __ldcg(Pp + s2 * kStride));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int s2 = 0; s2 < nsb; ++s2) {
      const float ms = __ldcg(Pp + s2 * kStride);
      if (ms == -INFINITY) continue;
      const float w = exp2f(ms - M);
      L = fmaf(w, __ldcg(Pp + s2 * kStride + 1), L);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        acc[e] = fmaf(w, __ldcg(Pp + s2 * kStride + 2 + 4 * lane + e), acc[e]);
    }
    const float il = L > 0.f ? 1.f / L : 0.f;
    __half2 o01 = __floats2half2_rn(acc[0] * il, acc[1] * il);
    __half2 o23 = __floats2half2_rn(acc[2] * il, acc[3] * il);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&o01);
    pk.y = *reinterpret_cast<uint32_t*>(&o23);
    *reinterpret_cast<uint2*>(ob + h * kD + 4 * lane) = pk;
  }
  if (lane == 0) a.ws_count[(int64_t)b * a.hkv + kvh] = 0;
}

template <int NT>
cudaError_t launch_nt(const DecodeArgs& a, cudaStream_t s) {
  static bool attr_set = false;
  const int smem = (int)sizeof(MmaSmem<NT>);
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<NT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(a.nsplit, a.hkv, a.batch);
  decode_mma_kernel<NT><<<grid, 32, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool decode_mma_supported(int g) { return g >= 1 && g <= 8; }

// Resident one-warp CTAs per SM, from the shared-memory footprint (228 KB per
// SM, 1 KB reserved per CTA).  Host-only arithmetic: no CUDA call.
int decode_mma_ctas_per_sm(int g) {
  const int bytes = g <= 4 ? (int)sizeof(MmaSmem<1>) : (int)sizeof(MmaSmem<2>);
  return 233472 / (bytes + 1024);
}

cudaError_t launch_decode_mma(const DecodeArgs& a, cudaStream_t s) {
  return a.g <= 4 ? launch_nt<1>(a, s) : launch_nt<2>(a, s);
}

}  // namespace kvarn
