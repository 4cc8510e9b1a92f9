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
// small integers with a query-side factor.  They run as mma.sync with the
// codes fed straight from the packed words: one AND leaves a code q at bit
// position 4i (K) or 2i (V) of each 16-bit half, which read as an fp16 is the
// subnormal q * 2^(4i-24) (resp. 2^(2i-24)), exact.  The power of two is
// undone on the query side, which is scaled by a power of two into range and
// split into an fp16 pair hi + lo, hi on a fixed grid (grid_hi below) so that
// the tensor core's fp32 sums of the hi products are exact.
//
// CTA = 4 warps, each an independent stream over the pages of its split of
// one (sequence, KV head): warp w takes pages u0 + w, u0 + w + 4, ...  Each
// warp double-buffers one 15360-byte page record in shared memory: the K part
// and the V part arrive by cp.async.bulk (TMA engine) on two mbarriers; the
// next page's K part loads while this page's values are summed, its V part
// while the next scores are computed.  The probabilities move from the score
// fragments to the value-sum fragments in registers (movmatrix transpose).
// Every wait is bounded; on expiry the warp reports KVARN_STATUS_TIMEOUT and
// drains its copies.  The four warps' softmax states are merged in shared
// memory, rotated back to plain space once per CTA, the split holding the end
// of the sequence adds the fp16 tail, and the splits of one (sequence, KV
// head) are merged (log-sum-exp) by the last CTA to arrive, in the same launch.
#include "kvarn_internal.cuh"
#include "ptx.cuh"

namespace kvarn {
namespace {

using namespace ptx;

constexpr int kWarps = 4;
// Largest split count merged inside a thread-block cluster; more splits merge
// through the workspace (partial states and arrival tickets).
constexpr int kMaxClusterSplits = 4;
constexpr int kThreads = 32 * kWarps;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kTwo24 = 16777216.0f;

// RB: the record format's bytes (RecFmt<FMT>::bytes)
template <int NT, int RB>
struct __align__(128) MmaSmem {
  uint8_t rec[kWarps][RB];       // per warp: K part at 0, V part at the format's kpart
  float qrot[4 * NT][kD];        // H q per (padded) query head of the group
  float qplain[4 * NT][kD];      // q itself, for the fp16 tail
  uint64_t bar[kWarps][2];       // per warp: 0 = K part landed, 1 = V part landed
  int ticket;
};
// row pitch (floats) of a warp's output state in its page buffer: rows 8 banks
// apart, so that the four heads (qi) of one store hit different banks
constexpr int kOPitch = kD + 8;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// fp16x2 with `first` in the low half
__device__ __forceinline__ uint32_t pack2(float first, float second) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(second), "f"(first));
  return r;
}

__device__ __forceinline__ uint32_t movm_trans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

// Split of an fp32 operand into two fp16 halves, hi + lo, for the tensor
// cores.  hi is x rounded to the nearest multiple of a fixed power of two g
// (adding and removing magic = 1.5 * 2^23 * g leaves the bits at and above g,
// for |x| < 2^22 g); lo = x - hi is exact in fp32 and |lo| <= g / 2.
//
// The grid is fixed per operand column rather than relative to each x.  On
// B300 an mma.sync with fp32 accumulation behaves as if it aligned its 16
// products to the largest one and dropped the bits more than about 16 bits
// below it: with an 11-significant-bit hi, sums of non-negative products came
// out low by ~1e-4 relative, the same on every channel.  With hi on a grid of
// g and |x| <= 2^11 g, every hi product is a multiple of g (codes are
// integers) and the 16 of them span about 13 bits, so the sum is exact; what
// the lo column can lose is at most ~2^-18 of the total.
__device__ __forceinline__ float grid_hi(float x, float magic) {
  return __fadd_rn(__fadd_rn(x, magic), -magic);
}
__device__ __forceinline__ float2 grid_hi2(float2 x, float magic) {   // both halves, one grid
  return __fadd2_rn(__fadd2_rn(x, make_float2(magic, magic)), make_float2(-magic, -magic));
}
constexpr float kMagic1 = 12582912.f;   // 1.5 * 2^23: magic for g = 1

// 2^k scale that maps amax into [2^14, 2^15), and its inverse.
__device__ __forceinline__ void pow2_scale(float amax, float& s, float& inv) {
  const int e = (__float_as_int(amax) >> 23) & 0xff;
  const int se = min(max(268 - e, 1), 253);
  s = __int_as_float(se << 23);
  inv = __int_as_float((254 - se) << 23);
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

// Position of channel ch in a row of qrot: the float4 index is XOR-ed with
// ch >> 5, so that the four lanes reading float4 k of their 32-channel slices
// (8 qi + k) hit four different bank groups.
__device__ __forceinline__ int qrot_pos(int ch) {
  return ((((ch >> 2) ^ (ch >> 5)) & 7) | ((ch >> 2) & ~7)) * 4 + (ch & 3);
}

__device__ __forceinline__ uint32_t word_of(const uint4& w, int i) {
  return i == 0 ? w.x : i == 1 ? w.y : i == 2 ? w.z : w.w;
}

// mask selecting crumb p (0..4) of both 16-bit halves
__device__ __forceinline__ constexpr uint32_t cmask(int p) { return 0x00030003u << (2 * p); }

// 1 / (power of two carried by the V code of a token in k-tile kb, half f)
__device__ __forceinline__ constexpr float vpos_inv(int kb, int f) {
  return (kb & 3) == 0 ? (f ? 0.25f : 1.f)
       : (kb & 3) == 1 ? (f ? 1.f / 64 : 1.f / 16)
       : (kb & 3) == 2 ? (f ? 1.f : 1.f / 256)
                       : (f ? 1.f / 16 : 0.25f);
}

// Three CTAs per SM for one head tile; for two (groups of 5-8 query heads)
// the doubled score, probability and accumulator fragments need more than the
// 168 registers a third CTA would leave, so two CTAs run with no spills.
// FMT: the record format (RecFmt).  A page token dequantizes as
// yhat_td = alpha_t beta_d q_td + gamma_t delta_d, so the score is
// alpha_t sum_d (q~_d beta_d) q_td + gamma_t sum_d q~_d delta_d and the value
// sum beta_d sum_t (p_t alpha_t) q_td + delta_d sum_t p_t gamma_t.
// The 27648-byte records of 8-bit keys leave shared memory for two CTAs per
// SM with one head tile and one with two, which may take every register.
template <int NT, int FMT>
__global__ void __launch_bounds__(kThreads, FMT == kFmtK8 ? 3 - NT : NT == 1 ? 3 : 2)
    decode_mma_kernel(DecodeArgs a) {
  using F = RecFmt<FMT>;
  constexpr int NG = F::g64 ? 2 : 1;     // channel groups with their own s', z'
  extern __shared__ __align__(128) uint8_t smem_raw[];
  MmaSmem<NT, F::bytes>& S = *reinterpret_cast<MmaSmem<NT, F::bytes>*>(smem_raw);
  constexpr int G = 4 * NT;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = lane >> 2, qi = lane & 3;
  const int g = a.g;
  const float sl2 = a.scale * kLog2e;   // scores are kept in log2 units

  int len = a.seq_lens[b];
  if (len < 0 || len > a.max_seq || len / kT > a.max_blocks) {
    if (split == 0 && kvh == 0 && tid == 0) report(a.status, KVARN_STATUS_BAD_LENGTH);
    len = 0;
  }
  const int nfull = len / kT, rem = len % kT;
  const int pps = a.pages_per_split;
  const int nsb = nfull > 0 ? (nfull + pps - 1) / pps : 1;
  // in a cluster every CTA takes part in the merge, with or without pages
  if (split >= nsb && !a.cluster) return;
  const int u0 = split * pps, u1 = min(nfull, u0 + pps);
  const bool has_tail = split == nsb - 1 && rem > 0;

  uint8_t* const kst = S.rec[warp];
  uint8_t* const vst = S.rec[warp] + F::kpart;
  uint64_t* const kbar = &S.bar[warp][0];
  uint64_t* const vbar = &S.bar[warp][1];
  if (lane == 0) {
    mbar_init(kbar, 1);
    mbar_init(vbar, 1);
    fence_mbar_init();
  }
  __syncwarp();

  const int32_t* trow = a.block_table + (int64_t)b * a.max_blocks;
  // page ids of this warp's pages u, u + 4, ... (32 of them from `ubase`, one
  // per lane); entries outside the pool are reported and skipped (-1)
  auto fetch_ids = [&](int ubase) -> int {
    const int uu = ubase + kWarps * lane;
    int p = -1;
    if (uu < u1) {
      p = trow[uu];
      if (p < 0 || (int64_t)p >= a.num_pages) {
        report(a.status, KVARN_STATUS_BAD_PAGE);
        p = -1;
      }
    }
    return p;
  };
  auto rec_of = [&](int64_t page) { return a.pool + (page * a.hkv + kvh) * (int64_t)F::bytes; };
  auto issue_k = [&](int64_t page) {
    if (lane == 0) {
      mbar_arrive_expect_tx(kbar, F::kpart);
      bulk_g2s(kst, rec_of(page), F::kpart, kbar);
    }
  };
  auto issue_v = [&](int64_t page) {
    if (lane == 0) {
      mbar_arrive_expect_tx(vbar, F::vpart);
      bulk_g2s(vst, rec_of(page) + F::kpart, F::vpart, vbar);
    }
  };

  // the query (warp w: heads w, w + 4; lane holds channels 32i + lane) and
  // this warp's page ids are fetched together
  const __half* qb = a.q + ((int64_t)b * a.hq + (int64_t)kvh * g) * kD;
  float xq[NT][4];
#pragma unroll
  for (int hh = 0; hh < NT; ++hh) {
    const int h = warp + kWarps * hh;
#pragma unroll
    for (int i = 0; i < 4; ++i) xq[hh][i] = h < g ? __half2float(qb[h * kD + 32 * i + lane]) : 0.f;
  }
  int u = u0 + warp;
  int ids = fetch_ids(u);
  int jb = 0;   // index of page u within the current batch of ids
  const __half* tkb = a.tail_k + ((int64_t)b * a.hkv + kvh) * kT * kD;
  const __half* tvb = a.tail_v + ((int64_t)b * a.hkv + kvh) * kT * kD;
  if (has_tail && warp == kWarps - 1 && lane == 0 &&
      ((reinterpret_cast<uintptr_t>(tkb) | reinterpret_cast<uintptr_t>(tvb)) & 15) == 0) {
    // the tail is read at the end: have it in L2 by then
    bulk_prefetch_l2(tkb, (uint32_t)rem * kD * 2);
    bulk_prefetch_l2(tvb, (uint32_t)rem * kD * 2);
  }

  // this warp's first page in flight while the query is rotated
  int64_t cur = __shfl_sync(0xffffffffu, ids, 0);
  bool k_busy = false, v_busy = false;
  uint32_t kph = 0, vph = 0;
  if (cur >= 0) {
    issue_k(cur);
    issue_v(cur);
    k_busy = v_busy = true;
  }

  // ---- q~ = H q ----
#pragma unroll
  for (int hh = 0; hh < NT; ++hh) {
    const int h = warp + kWarps * hh;
    float* x = xq[hh];
#pragma unroll
    for (int i = 0; i < 4; ++i) S.qplain[h][32 * i + lane] = x[i] * sl2;
    // channel bits 5, 6 are local
    float y0 = x[0] + x[1], y1 = x[0] - x[1], y2 = x[2] + x[3], y3 = x[2] - x[3];
    x[0] = y0 + y2; x[2] = y0 - y2; x[1] = y1 + y3; x[3] = y1 - y3;
    // channel bits 0..4 across lanes
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      const bool up = lane & m;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float o = __shfl_xor_sync(0xffffffffu, x[i], m);
        x[i] = up ? o - x[i] : x[i] + o;
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) S.qrot[h][qrot_pos(32 * i + lane)] = x[i] * kInvSqrt128;
  }
  __syncthreads();

  float m[NT], l[NT], oacc[NT][16];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m[nt] = -INFINITY;
    l[nt] = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) oacc[nt][j] = 0.f;
  }
  bool timed_out = false;

  for (; u < u1; u += kWarps) {
    float sc[NT][16];
    if (cur >= 0) {
      if (!mbar_wait_warp(kbar, kph, kWaitLimitNs)) {
        timed_out = true;
        break;
      }
      kph ^= 1;
      k_busy = false;

      // ---- per channel group (one for the per-token formats, two for g64,
      // whose groups of 64 channels carry their own s', z'): query-side B
      // fragments, then the scores of the group's k-tiles ----
      // B fragments: qc = q~ * beta^K, scaled, split hi / lo.  B column n = r:
      // head 4nt + (r >> 1), hi part (r even) or lo part (r odd); k rows 2qi..
      // of k-tile kb hold channels g0 + c0, c0 + 4 with g0 the lane's first
      // channel of the group (32 qi; for g64 64 gi + 16 qi) and
      // c0 = 8 (kb >> 1) + 2 (kb & 1) + slot.  The slot-1 channels meet codes
      // carrying 16x (nibble at bits 4-7) and are pre-scaled by 1/16.
      constexpr int KB = 8 / NG;             // k-tiles per group
      constexpr int CPL = 32 / NG;           // channels per lane per group
      const bool odd = r & 1;
#pragma unroll
      for (int gi = 0; gi < NG; ++gi) {
        uint32_t bq[NT][KB][2];
        float sA[NT], sZ[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int h = 4 * nt + (r >> 1);
          const float4* qv = reinterpret_cast<const float4*>(S.qrot[h]);
          const uint8_t* cv = kst + F::kc;   // beta, delta of the lane's channels
          float v[CPL];
          float am0 = 0.f, am1 = 0.f;
          float2 s0 = make_float2(0.f, 0.f), s1 = s0;
#pragma unroll
          for (int k = 0; k < CPL / 4; ++k) {
            const int ch = (NG == 1 ? 32 * qi : 64 * gi + 16 * qi) + 4 * k;
            const int idx = ch >> 2;
            const float4 q4 = qv[((idx ^ (ch >> 5)) & 7) | (idx & ~7)];   // qrot_pos
            const float4 c4 = F::get_b4(cv, idx);
            const float2 p0 = __fmul2_rn(make_float2(q4.x, q4.y), make_float2(c4.x, c4.y));
            const float2 p1 = __fmul2_rn(make_float2(q4.z, q4.w), make_float2(c4.z, c4.w));
            v[4 * k + 0] = p0.x;
            v[4 * k + 1] = p0.y;
            v[4 * k + 2] = p1.x;
            v[4 * k + 3] = p1.y;
            am0 = max3(am0, fabsf(p0.x), fabsf(p0.y));
            am1 = max3(am1, fabsf(p1.x), fabsf(p1.y));
            if constexpr (F::pc) {   // the constant term takes delta, not beta
              const float4 d4 = F::get_d4(cv, idx);
              s0 = __ffma2_rn(make_float2(q4.x, q4.y), make_float2(d4.x, d4.y), s0);
              s1 = __ffma2_rn(make_float2(q4.z, q4.w), make_float2(d4.z, d4.w), s1);
            } else {
              s0 = __fadd2_rn(s0, p0);
              s1 = __fadd2_rn(s1, p1);
            }
          }
          float amax = fmaxf(am0, am1);
          const float2 s01 = __fadd2_rn(s0, s1);
          float sum = s01.x + s01.y;
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
          sum += __shfl_xor_sync(0xffffffffu, sum, 1);
          sum += __shfl_xor_sync(0xffffffffu, sum, 2);
          float scl, inv;
          pow2_scale(amax, scl, inv);
          const float scl16 = scl * 0.0625f;
#pragma unroll
          for (int kb = 0; kb < KB; ++kb) {
#pragma unroll
            for (int slot = 0; slot < 2; ++slot) {
              // 8-bit codes (bytes 4 (kb & 3) .. of the lane's 16-byte chunk
              // kb >> 2): k rows 2qi, 2qi + 1 | 2qi + 8, 2qi + 9 hold
              // channels 4 kb + 2 slot + 0, 1, both at bit 0 of their half
              const int c0 = F::k8 ? 4 * kb + 2 * slot : 8 * (kb >> 1) + 2 * (kb & 1) + slot;
              const int c1 = F::k8 ? c0 + 1 : c0 + 4;
              const float f = slot && !F::k8 ? scl16 : scl;
              // |x| < 2^15 (slot 0) or 2^11 (slot 1): grid 16 or 1, i.e. 16
              // in the units of the 4-bit code it meets; for 8-bit codes
              // grid 256, so that a hi product spans 15 bits as with 4-bit
              const float2 x = __fmul2_rn(make_float2(v[c0], v[c1]), make_float2(f, f));
              const float2 hg =
                  grid_hi2(x, F::k8 ? 256.f * kMagic1 : slot ? kMagic1 : 16.f * kMagic1);
              const float2 o = odd ? __ffma2_rn(hg, make_float2(-1.f, -1.f), x) : hg;   // lo | hi
              bq[nt][kb][slot] = pack2(o.x, o.y);
            }
          }
          // this lane's score column pair (2qi, 2qi+1) is head 4nt + qi, held
          // by lanes with r = 2qi: fetch that head's scale and sum
          sA[nt] = __shfl_sync(0xffffffffu, inv, 8 * qi) * (kTwo24 * sl2);
          sZ[nt] = __shfl_sync(0xffffffffu, sum, 8 * qi) * sl2;
        }

        // ---- scores: K codes (A, rows = tokens) x qc (B).  MTG token tiles
        // at a time, k-tile outer, so that MTG accumulator chains interleave.
        // The lane's code words of a token row: 4 words at 16 qi (one group)
        // or 2 words at 32 gi + 8 qi (g64); 8-bit codes: its 16-byte chunks
        // 2qi, 2qi + 1 (k8_byte), one per half of the k-tiles ----
        constexpr int MTG = NT == 1 ? 8 : 4;
        constexpr int NH = F::k8 ? 2 : 1;
#pragma unroll
        for (int m0 = 0; m0 < 8; m0 += MTG) {
          float d[NT][MTG][4];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < MTG; ++i) d[nt][i][0] = d[nt][i][1] = d[nt][i][2] = d[nt][i][3] = 0.f;
#pragma unroll
          for (int hk = 0; hk < NH; ++hk) {
            uint4 kw[MTG][2];
#pragma unroll
            for (int i = 0; i < MTG; ++i) {
              const int tA = 16 * (m0 + i) + r;
              if constexpr (F::k8) {
                const int ofs = 16 * ((2 * qi + hk) ^ (r & 1));   // tA, tA + 8: parity of r
                kw[i][0] = *reinterpret_cast<const uint4*>(kst + 128 * tA + ofs);
                kw[i][1] = *reinterpret_cast<const uint4*>(kst + 128 * (tA + 8) + ofs);
              } else if constexpr (NG == 1) {
                kw[i][0] = *reinterpret_cast<const uint4*>(kst + kOffKCodes + 64 * tA + 16 * qi);
                kw[i][1] =
                    *reinterpret_cast<const uint4*>(kst + kOffKCodes + 64 * (tA + 8) + 16 * qi);
              } else {
                const uint2 wA = *reinterpret_cast<const uint2*>(kst + 64 * tA + 32 * gi + 8 * qi);
                const uint2 wB =
                    *reinterpret_cast<const uint2*>(kst + 64 * (tA + 8) + 32 * gi + 8 * qi);
                kw[i][0] = make_uint4(wA.x, wA.y, 0u, 0u);
                kw[i][1] = make_uint4(wB.x, wB.y, 0u, 0u);
              }
            }
#pragma unroll
            for (int kk = 0; kk < KB / NH; ++kk) {
              const int kb = (KB / NH) * hk + kk;
#pragma unroll
              for (int i = 0; i < MTG; ++i) {
                uint32_t A[4];
                if constexpr (F::k8) {
                  // bytes 0, 1 (a0, a1) and 2, 3 (a2, a3) of word kk, each
                  // moved to bit 0 of a 16-bit half
                  const uint32_t wa = word_of(kw[i][0], kk), wb = word_of(kw[i][1], kk);
                  A[0] = __byte_perm(wa, 0u, 0x4140);
                  A[1] = __byte_perm(wb, 0u, 0x4140);
                  A[2] = __byte_perm(wa, 0u, 0x4342);
                  A[3] = __byte_perm(wb, 0u, 0x4342);
                } else {
                  uint32_t wa = word_of(kw[i][0], kb >> 1), wb = word_of(kw[i][1], kb >> 1);
                  if (kb & 1) {
                    wa >>= 8;
                    wb >>= 8;
                  }
                  A[0] = wa & 0x000F000Fu;
                  A[1] = wb & 0x000F000Fu;
                  A[2] = wa & 0x00F000F0u;
                  A[3] = wb & 0x00F000F0u;
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                  mma_16816(d[nt][i], A, bq[nt][kb][0], bq[nt][kb][1]);
              }
            }
          }
#pragma unroll
          for (int i = 0; i < MTG; ++i) {
            const int mt = m0 + i, tA = 16 * mt + r, tB = tA + 8;
            const float2 szA = F::get_sz_g(kst + F::ksz, tA, gi);
            const float2 szB = F::get_sz_g(kst + F::ksz, tB, gi);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const float xA = fmaf(szA.x * sA[nt], d[nt][i][0] + d[nt][i][1], szA.y * sZ[nt]);
              const float xB = fmaf(szB.x * sA[nt], d[nt][i][2] + d[nt][i][3], szB.y * sZ[nt]);
              sc[nt][2 * mt] = gi == 0 ? xA : sc[nt][2 * mt] + xA;
              sc[nt][2 * mt + 1] = gi == 0 ? xB : sc[nt][2 * mt + 1] + xB;
            }
          }
        }
      }
    }
    __syncwarp();   // the K part of this page is consumed
    if (++jb == 32) {
      ids = fetch_ids(u + kWarps);
      jb = 0;
    }
    const int64_t nxt = __shfl_sync(0xffffffffu, ids, jb);
    if (nxt >= 0) {
      issue_k(nxt);
      k_busy = true;
    }
    if (cur >= 0) {
      // ---- online softmax (log2 units); l is a per-lane partial sum ----
      float alpha[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float pq[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          pq[k] = fmaxf(max3(sc[nt][4 * k], sc[nt][4 * k + 1], sc[nt][4 * k + 2]), sc[nt][4 * k + 3]);
        float pm = fmaxf(max3(pq[0], pq[1], pq[2]), pq[3]);
        pm = warp_max_r(pm);
        const float mnew = fmaxf(m[nt], pm);
        alpha[nt] = ex2(m[nt] - mnew);
        m[nt] = mnew;
        float lq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          sc[nt][j] = ex2(sc[nt][j] - mnew);   // now p
          lq[j & 3] += sc[nt][j];
        }
        l[nt] = fmaf(l[nt], alpha[nt], (lq[0] + lq[1]) + (lq[2] + lq[3]));
      }

      if (!mbar_wait_warp(vbar, vph, kWaitLimitNs)) {
        timed_out = true;
        break;
      }
      vph ^= 1;
      v_busy = false;

      // ---- per channel group (two for g64): P' = p s'V (scaled, hi | lo)
      // transposed into B fragments, then the value sums of the group's
      // channel tiles (16 channels each; channels 64 gi .. for g64) ----
      // score slot j of this lane is token 16 (j >> 1) + 8 (j & 1) + r
      const uint8_t* cvv = vst + (F::vc - F::kpart);
#pragma unroll
      for (int gi = 0; gi < NG; ++gi) {
        float2 szv[16];
        float sm4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          szv[j] = F::get_sz_g(vst + (F::vsz - F::kpart), 16 * (j >> 1) + 8 * (j & 1) + r, gi);
          sm4[j & 3] = fmaxf(sm4[j & 3], szv[j].x);
        }
        float smax = fmaxf(fmaxf(sm4[0], sm4[1]), fmaxf(sm4[2], sm4[3]));
        smax = warp_max_r(smax);
        float fs, finv;
        pow2_scale(smax, fs, finv);
        float sf[16];
        // 1 / (power of two carried by the V code of score slot j): the 2-bit
        // crumb positions, or for 4-bit codes nibble 0 (k rows 0-7) or 1 (x16)
        auto pos_inv = [](int kb, int f) { return F::v4 ? (f ? 0.0625f : 1.f) : vpos_inv(kb, f); };
#pragma unroll
        for (int j = 0; j < 16; ++j) sf[j] = szv[j].x * (fs * pos_inv(j >> 1, j & 1));
        uint32_t bp[NT][8][2];
        float zpage[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float zq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            // x <= 2^15 / 4^pos for a code carrying 4^pos: grid 16 / 4^pos
            const float x = sc[nt][j] * sf[j];
            const float hi = grid_hi(x, (16.f * kMagic1) * pos_inv(j >> 1, j & 1));
            bp[nt][j >> 1][j & 1] = movm_trans(pack2(hi, x - hi));
            zq[j & 3] = fmaf(sc[nt][j], szv[j].y, zq[j & 3]);
          }
          zpage[nt] = warp_sum_r((zq[0] + zq[1]) + (zq[2] + zq[3]));
        }

        // ---- value sum: V codes (A, rows = channels) x P' (B).  MCG channel
        // tiles at a time, k-tile outer, so that their chains interleave ----
        const float fin = finv * kTwo24;
        constexpr int MCG = (NT == 1 ? 8 : 4) / NG / (F::v4 ? 2 : 1);
#pragma unroll
        for (int c0 = 8 * gi / NG; c0 < 8 * (gi + 1) / NG; c0 += MCG) {
          // 2-bit: words (e, h) = 00, 01, 10, 11 of channels 16mc + r, + 8.
          // 4-bit: words p = 0..3 of channel 16mc + r (vw) and of 16mc + 8 + r
          // (vw4), v4_word(c, lane & 3, p)
          uint4 vw[MCG], vw4[F::v4 ? MCG : 1];
#pragma unroll
          for (int i = 0; i < MCG; ++i) {
            if constexpr (F::v4) {
              vw[i] = *reinterpret_cast<const uint4*>(vst + 1024 * (c0 + i) + 32 * lane);
              vw4[i] = *reinterpret_cast<const uint4*>(vst + 1024 * (c0 + i) + 32 * lane + 16);
            } else {
              vw[i] = *reinterpret_cast<const uint4*>(vst + 512 * (c0 + i) + 16 * lane);
            }
          }
          float d[NT][MCG][4];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < MCG; ++i) d[nt][i][0] = d[nt][i][1] = d[nt][i][2] = d[nt][i][3] = 0.f;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              const int kb = 4 * hh + jj;
#pragma unroll
              for (int i = 0; i < MCG; ++i) {
                uint32_t A[4];
                if constexpr (F::v4) {
                  // k-tile kb: word kb >> 1, nibbles 0, 4 (a0, a1) and 1, 5
                  // (a2, a3; x16) after a shift by 8 for odd kb
                  uint32_t w0 = word_of(vw[i], kb >> 1), w1 = word_of(vw4[i], kb >> 1);
                  if (kb & 1) {
                    w0 >>= 8;
                    w1 >>= 8;
                  }
                  A[0] = w0 & 0x000F000Fu; A[1] = w1 & 0x000F000Fu;
                  A[2] = w0 & 0x00F000F0u; A[3] = w1 & 0x00F000F0u;
#pragma unroll
                  for (int nt = 0; nt < NT; ++nt) mma_16816(d[nt][i], A, bp[nt][kb][0], bp[nt][kb][1]);
                  continue;
                }
                const uint32_t e0 = word_of(vw[i], hh), e1 = word_of(vw[i], 2 + hh);
                if (jj == 0) {
                  A[0] = e0 & cmask(0); A[1] = e1 & cmask(0); A[2] = e0 & cmask(1); A[3] = e1 & cmask(1);
                } else if (jj == 1) {
                  A[0] = e0 & cmask(2); A[1] = e1 & cmask(2); A[2] = e0 & cmask(3); A[3] = e1 & cmask(3);
                } else if (jj == 2) {
                  A[0] = e0 & cmask(4); A[1] = e1 & cmask(4);
                  A[2] = (e0 >> 10) & cmask(0); A[3] = (e1 >> 10) & cmask(0);
                } else {
                  A[0] = (e0 >> 10) & cmask(1); A[1] = (e1 >> 10) & cmask(1);
                  A[2] = (e0 >> 10) & cmask(2); A[3] = (e1 >> 10) & cmask(2);
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) mma_16816(d[nt][i], A, bp[nt][kb][0], bp[nt][kb][1]);
              }
            }
          }
#pragma unroll
          for (int i = 0; i < MCG; ++i) {
            const int mc = c0 + i;
            const float2 bdA = F::get_bd(cvv, 16 * mc + r), bdB = F::get_bd(cvv, 16 * mc + 8 + r);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              float uA, uB;
              if constexpr (F::pc) {
                uA = fmaf(bdA.x, (d[nt][i][0] + d[nt][i][1]) * fin, bdA.y * zpage[nt]);
                uB = fmaf(bdB.x, (d[nt][i][2] + d[nt][i][3]) * fin, bdB.y * zpage[nt]);
              } else {   // beta = delta = c
                uA = bdA.x * fmaf(d[nt][i][0] + d[nt][i][1], fin, zpage[nt]);
                uB = bdB.x * fmaf(d[nt][i][2] + d[nt][i][3], fin, zpage[nt]);
              }
              oacc[nt][2 * mc] = fmaf(oacc[nt][2 * mc], alpha[nt], uA);
              oacc[nt][2 * mc + 1] = fmaf(oacc[nt][2 * mc + 1], alpha[nt], uB);
            }
          }
        }
      }
    }
    __syncwarp();   // the V part of this page is consumed
    if (nxt >= 0) {
      issue_v(nxt);
      v_busy = true;
    }
    cur = nxt;
  }

  if (timed_out) {
    if (lane == 0) report(a.status, KVARN_STATUS_TIMEOUT);
    // drain copies still in flight before the buffer is reused or released
    if (k_busy) mbar_wait_bounded(kbar, kph, kWaitLimitNs);
    if (v_busy) mbar_wait_bounded(vbar, vph, kWaitLimitNs);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m[nt] = -INFINITY;
      l[nt] = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) oacc[nt][j] = 0.f;
    }
  }
  __syncwarp();

  // ---- back to plain space, in registers: lane (r, qi) holds for head
  // 4nt + qi the channels 16 mc + 8 e + r at oacc[nt][2 mc + e], so channel
  // bits 3..6 are local and bits 0..2 are lane bits 2..4 ----
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float* o = oacc[nt];
#pragma unroll
    for (int hb = 1; hb < 16; hb <<= 1)
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if ((j & hb) == 0) {
          const float x = o[j], y = o[j + hb];
          o[j] = x + y;
          o[j + hb] = x - y;
        }
#pragma unroll
    for (int lb = 4; lb < 32; lb <<= 1) {
      const bool up = lane & lb;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float other = __shfl_xor_sync(0xffffffffu, o[j], lb);
        o[j] = up ? other - o[j] : o[j] + other;
      }
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) o[j] *= kInvSqrt128;
  }

  // ---- this warp's state into its own buffer: [G]{m, l}, then o[G][kOPitch] ----
  float* st = reinterpret_cast<float*>(kst);
  float* ow = st + 2 * G;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const float lsum = warp_sum_r(l[nt]);
#pragma unroll
    for (int mc = 0; mc < 8; ++mc) {
      ow[(4 * nt + qi) * kOPitch + 16 * mc + r] = oacc[nt][2 * mc];
      ow[(4 * nt + qi) * kOPitch + 16 * mc + 8 + r] = oacc[nt][2 * mc + 1];
    }
    if (r == 0) {
      st[2 * (4 * nt + qi)] = m[nt];
      st[2 * (4 * nt + qi) + 1] = lsum;
    }
  }
  __syncwarp();

  // ---- fp16 tail (plain space): warp w takes tail tokens 3 - w, 7 - w, ...
  // and folds them into its own state; lane holds channels 4 lane .. + 3 ----
  if (has_tail && !timed_out) {
    float qr[G][4], mt[G], lt[G], ot[G][4];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float4 q4 = *reinterpret_cast<const float4*>(&S.qplain[h][4 * lane]);
      qr[h][0] = q4.x;
      qr[h][1] = q4.y;
      qr[h][2] = q4.z;
      qr[h][3] = q4.w;
      mt[h] = st[2 * h];
      lt[h] = st[2 * h + 1];
      const float4 o4 = *reinterpret_cast<const float4*>(ow + h * kOPitch + 4 * lane);
      ot[h][0] = o4.x;
      ot[h][1] = o4.y;
      ot[h][2] = o4.z;
      ot[h][3] = o4.w;
    }
    constexpr int kC = 8;   // tail tokens per batch of loads
    // warp w takes tail tokens from kWarps - 1 - w: the higher warps of a split
    // hold no more pages than the lower ones
    for (int t0 = kWarps - 1 - warp; t0 < rem; t0 += kWarps * kC) {
      uint2 kk[kC], vv[kC];
#pragma unroll
      for (int i = 0; i < kC; ++i) {
        const int t = t0 + kWarps * i;
        if (t < rem) {
          kk[i] = __ldg(reinterpret_cast<const uint2*>(tkb + (int64_t)t * kD + 4 * lane));
          vv[i] = __ldg(reinterpret_cast<const uint2*>(tvb + (int64_t)t * kD + 4 * lane));
        }
      }
#pragma unroll
      for (int i = 0; i < kC; ++i) {
        if (t0 + kWarps * i >= rem) break;
        const float2 k01 = __half22float2(*reinterpret_cast<const __half2*>(&kk[i].x));
        const float2 k23 = __half22float2(*reinterpret_cast<const __half2*>(&kk[i].y));
        const float2 v01 = __half22float2(*reinterpret_cast<const __half2*>(&vv[i].x));
        const float2 v23 = __half22float2(*reinterpret_cast<const __half2*>(&vv[i].y));
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float sc1 = fmaf(qr[h][0], k01.x, fmaf(qr[h][1], k01.y,
                      fmaf(qr[h][2], k23.x, qr[h][3] * k23.y)));
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) sc1 += __shfl_xor_sync(0xffffffffu, sc1, o);
          const float mn = fmaxf(mt[h], sc1);
          const float al = ex2(mt[h] - mn), pt = ex2(sc1 - mn);
          mt[h] = mn;
          lt[h] = fmaf(lt[h], al, pt);
          ot[h][0] = fmaf(ot[h][0], al, pt * v01.x);
          ot[h][1] = fmaf(ot[h][1], al, pt * v01.y);
          ot[h][2] = fmaf(ot[h][2], al, pt * v23.x);
          ot[h][3] = fmaf(ot[h][3], al, pt * v23.y);
        }
      }
    }
    __syncwarp();
#pragma unroll
    for (int h = 0; h < G; ++h) {
      if (lane == 0) {
        st[2 * h] = mt[h];
        st[2 * h + 1] = lt[h];
      }
      *reinterpret_cast<float4*>(ow + h * kOPitch + 4 * lane) =
          make_float4(ot[h][0], ot[h][1], ot[h][2], ot[h][3]);
    }
  }
  __syncthreads();

  // ---- merge the warps' states; the result goes straight to the output
  // (one split), to shared memory for the cluster merge, or to this split's
  // partial state ----
  __half* ob = a.out + ((int64_t)b * a.hq + (int64_t)kvh * g) * kD;
  if (a.cluster) {
    // CTA state in registers (thread: entries tid, tid + 128, ...), then in
    // warp 0's buffer as [G]{M, L}, o[G][kD]
    constexpr int kPer = G * kD / kThreads;
    float cM[kPer], cL[kPer], cO[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = tid + kThreads * k, h = i >> 7, ch = i & 127;
      float M = -INFINITY, o = 0.f, L = 0.f;
      if (h < g) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
          M = fmaxf(M, reinterpret_cast<const float*>(S.rec[w])[2 * h]);
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kWarps; ++w) {
            const float* sw = reinterpret_cast<const float*>(S.rec[w]);
            const float wt = ex2(sw[2 * h] - M);
            o = fmaf(wt, sw[2 * G + h * kOPitch + ch], o);
            L = fmaf(wt, sw[2 * h + 1], L);
          }
        }
      }
      cM[k] = M;
      cL[k] = L;
      cO[k] = o;
    }
    __syncthreads();
    float* cs = reinterpret_cast<float*>(S.rec[0]);
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = tid + kThreads * k, h = i >> 7, ch = i & 127;
      if (ch == 0) {
        cs[2 * h] = cM[k];
        cs[2 * h + 1] = cL[k];
      }
      cs[2 * G + i] = cO[k];
    }
    cluster_sync();
    if (cluster_ctarank() == 0) {
      // rank 0 merges the cluster's states (distributed shared memory); a
      // thread's remote loads are all issued before the first is used
      const uint32_t nc = (uint32_t)a.nsplit;
#pragma unroll
      for (int k0 = 0; k0 < kPer; k0 += 4) {
        float Mr[4][kMaxClusterSplits], Lr[4][kMaxClusterSplits], Or[4][kMaxClusterSplits];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i = tid + kThreads * (k0 + k), h = i >> 7;
#pragma unroll
          for (uint32_t c = 0; c < (uint32_t)kMaxClusterSplits; ++c) {
            Mr[k][c] = -INFINITY;
            Lr[k][c] = Or[k][c] = 0.f;
            if (h < g && c < nc) {
              Mr[k][c] = ld_dsmem_f32(cs + 2 * h, c);
              Lr[k][c] = ld_dsmem_f32(cs + 2 * h + 1, c);
              Or[k][c] = ld_dsmem_f32(cs + 2 * G + i, c);
            }
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int i = tid + kThreads * (k0 + k), h = i >> 7;
          if (h >= g) continue;
          float M = -INFINITY;
#pragma unroll
          for (int c = 0; c < kMaxClusterSplits; ++c) M = fmaxf(M, Mr[k][c]);
          float o = 0.f, L = 0.f;
          if (M != -INFINITY) {
#pragma unroll
            for (int c = 0; c < kMaxClusterSplits; ++c) {
              const float wt = ex2(Mr[k][c] - M);   // 0 for an empty state
              o = fmaf(wt, Or[k][c], o);
              L = fmaf(wt, Lr[k][c], L);
            }
          }
          ob[i] = __float2half_rn(L > 0.f ? o / L : 0.f);
        }
      }
    }
    // no CTA leaves while rank 0 may still read its shared memory
    cluster_sync();
    return;
  }
  for (int i = tid; i < g * kD; i += kThreads) {
    const int h = i >> 7, ch = i & 127;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
      M = fmaxf(M, reinterpret_cast<const float*>(S.rec[w])[2 * h]);
    float o = 0.f, L = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float* sw = reinterpret_cast<const float*>(S.rec[w]);
        const float wt = ex2(sw[2 * h] - M);
        o = fmaf(wt, sw[2 * G + h * kOPitch + ch], o);
        L = fmaf(wt, sw[2 * h + 1], L);
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

  // ---- last split to arrive: merge all splits, warp w takes heads w, w + 4;
  // lane holds channels 4 lane .. + 3; loads batched kU splits deep ----
  for (int h = warp; h < g; h += kWarps) {
    const float* P0 = a.ws_part + (((int64_t)b * a.hq + kvh * g + h) * a.nsplit) * kPartStride;
    float M = -INFINITY, L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    constexpr int kU = 8;
    for (int s0 = 0; s0 < nsb; s0 += kU) {
      float2 ml[kU];
      float4 os[kU];
#pragma unroll
      for (int k = 0; k < kU; ++k) {
        if (s0 + k < nsb) {
          const float* Ps = P0 + (int64_t)(s0 + k) * kPartStride;
          ml[k] = __ldcg(reinterpret_cast<const float2*>(Ps));
          os[k] = __ldcg(reinterpret_cast<const float4*>(Ps + 4) + lane);
        } else {
          ml[k] = make_float2(-INFINITY, 0.f);
          os[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int k = 0; k < kU; ++k) {
        if (ml[k].x == -INFINITY) continue;
        const float Mn = fmaxf(M, ml[k].x);
        const float al = ex2(M - Mn), wt = ex2(ml[k].x - Mn);
        L = fmaf(L, al, wt * ml[k].y);
        acc.x = fmaf(acc.x, al, wt * os[k].x);
        acc.y = fmaf(acc.y, al, wt * os[k].y);
        acc.z = fmaf(acc.z, al, wt * os[k].z);
        acc.w = fmaf(acc.w, al, wt * os[k].w);
        M = Mn;
      }
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

template <int NT, int FMT>
cudaError_t launch_nt(const DecodeArgs& args, cudaStream_t s) {
  static std::atomic<uint64_t> smem_set{0};
  const int smem = (int)sizeof(MmaSmem<NT, RecFmt<FMT>::bytes>);
  cudaError_t e = ensure_dynamic_smem(decode_mma_kernel<NT, FMT>, smem, smem_set);
  if (e != cudaSuccess) return e;
  const DecodeArgs& a = args;   // a.cluster: the plan's choice of merge
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.nsplit, a.hkv, a.batch);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (a.cluster) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = a.nsplit;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, decode_mma_kernel<NT, FMT>, a);
}

}  // namespace

bool decode_mma_supported(int g) { return g >= 1 && g <= 8; }

int decode_mma_warps() { return kWarps; }

int decode_mma_max_cluster() { return kMaxClusterSplits; }

// CTAs per SM of one planned wave: at most what the shared-memory footprint
// (228 KB per SM, 1 KB reserved per CTA) and the launch bounds allow.
// Host-only arithmetic: no CUDA call.
// The split plan sizes one wave by this count.  Two CTAs per SM are planned
// even where three fit (one head tile): the plan then cuts each (sequence,
// KV head) into fewer, longer splits, whose per-CTA prologue and merge
// weigh less (the Llama-like layer decodes in 20.8 us instead of 21.7).  A
// grid larger than a wave still runs three per SM where they fit.
template <int RB>
int ctas_for(int g) {
  const int bytes = g <= 4 ? (int)sizeof(MmaSmem<1, RB>) : (int)sizeof(MmaSmem<2, RB>);
  return min(233472 / (bytes + 1024), 2);
}

// CTAs per SM that can be resident at once: the shared-memory footprint and
// the launch bounds (the register budget), without the plan's cap of two.
template <int RB, int FMT>
int resident_for(int g) {
  const int nt = g <= 4 ? 1 : 2;
  const int bytes = nt == 1 ? (int)sizeof(MmaSmem<1, RB>) : (int)sizeof(MmaSmem<2, RB>);
  const int lb = FMT == kFmtK8 ? 3 - nt : nt == 1 ? 3 : 2;
  return min(233472 / (bytes + 1024), lb);
}

int decode_mma_resident_per_sm(int g, int fmt) {
  switch (fmt) {
    case kFmtM16: return resident_for<RecFmt<kFmtM16>::bytes, kFmtM16>(g);
    case kFmtG64: return resident_for<RecFmt<kFmtG64>::bytes, kFmtG64>(g);
    case kFmtV4: return resident_for<RecFmt<kFmtV4>::bytes, kFmtV4>(g);
    case kFmtK8: return resident_for<RecFmt<kFmtK8>::bytes, kFmtK8>(g);
    default: return resident_for<RecFmt<kFmtF32>::bytes, kFmtF32>(g);
  }
}

int decode_mma_ctas_per_sm(int g, int fmt) {
  switch (fmt) {
    case kFmtM16: return ctas_for<RecFmt<kFmtM16>::bytes>(g);
    case kFmtG64: return ctas_for<RecFmt<kFmtG64>::bytes>(g);
    case kFmtV4: return ctas_for<RecFmt<kFmtV4>::bytes>(g);
    case kFmtK8: return ctas_for<RecFmt<kFmtK8>::bytes>(g);
    default: return ctas_for<RecFmt<kFmtF32>::bytes>(g);   // fp32 and per-channel records
  }
}

cudaError_t launch_decode_mma(const DecodeArgs& a, cudaStream_t s) {
  if (a.fmt == kFmtM16) return a.g <= 4 ? launch_nt<1, kFmtM16>(a, s) : launch_nt<2, kFmtM16>(a, s);
  if (a.fmt == kFmtPC) return a.g <= 4 ? launch_nt<1, kFmtPC>(a, s) : launch_nt<2, kFmtPC>(a, s);
  if (a.fmt == kFmtG64) return a.g <= 4 ? launch_nt<1, kFmtG64>(a, s) : launch_nt<2, kFmtG64>(a, s);
  if (a.fmt == kFmtV4) return a.g <= 4 ? launch_nt<1, kFmtV4>(a, s) : launch_nt<2, kFmtV4>(a, s);
  if (a.fmt == kFmtK8) return a.g <= 4 ? launch_nt<1, kFmtK8>(a, s) : launch_nt<2, kFmtK8>(a, s);
  return a.g <= 4 ? launch_nt<1, kFmtF32>(a, s) : launch_nt<2, kFmtF32>(a, s);
}

}  // namespace kvarn
