// decode_simple.cu -- paged split-K decode attention over the quantized cache,
// plain CUDA-core formulation (one thread per token for scores, one thread per
// channel for the value sum).  It is the reference CUDA path used for small
// GQA groups and as the fallback for configurations the tensor-core kernel
// does not cover.
//
// Method: one new query token per sequence attends to every cached token
// ("KV Cache (Anahtar-Deger Onbellegi)", yapayzekasozluk.tr, "KV Cache Nasil
// Calisir?").  Keys and values are stored rotated, y = H x, with H the
// orthonormal Hadamard matrix (KVarN page, blog.edumints.com, "KVarN Nasil
// Calisir?", stage "Dondurulmus Onbellek", which notes that the rotation keeps
// attention scores).  So the query is rotated once, q~ = H q, scores are taken
// against the rotated keys, the value sum is accumulated in rotated space and
// rotated back once at the end: o = H o~ + o_tail, the fp16 tail being added
// in plain space.  With the stored metadata,
//   q~ . yhat_t = s'_t * sum_d (q~_d c_d) q_td + z'_t * sum_d q~_d c_d.
#include "kvarn_internal.cuh"

namespace kvarn {
namespace {

constexpr int kThreads = 128;

struct __align__(16) DecodeSmem {
  uint8_t rec[kRecMax];
  float qrot[kMaxG][kD];   // H q, per head
  float qraw[kMaxG][kD];   // q, per head (tail scores)
  float qc[kMaxG][kD];     // H q * c^K, per page
  float pw[kMaxG][kT];     // p_t * s'^V_t, per page
  float pw1[kMaxG][kT];    //   of the second channel group (g64)
  float red[kThreads / 32][kMaxG];
  float m[kMaxG], l[kMaxG], alpha[kMaxG], sq[kMaxG], zs[kMaxG], sq1[kMaxG], zs1[kMaxG];
  int ticket;
};

// Block-wide reductions over the 128 threads, one value per head.
template <bool kMax>
__device__ __forceinline__ void block_reduce(DecodeSmem& S, float (&v)[kMaxG], int g,
                                             float* out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int h = 0; h < g; ++h) {
    float x = v[h];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      float y = __shfl_xor_sync(0xffffffffu, x, o);
      x = kMax ? fmaxf(x, y) : x + y;
    }
    if (lane == 0) S.red[warp][h] = x;
  }
  __syncthreads();
  if (threadIdx.x < g) {
    const int h = threadIdx.x;
    float x = S.red[0][h];
    for (int w = 1; w < kThreads / 32; ++w) x = kMax ? fmaxf(x, S.red[w][h]) : x + S.red[w][h];
    out[h] = x;
  }
  __syncthreads();
}

// In-place Walsh-Hadamard transform of g vectors of 128 floats, scaled.
__device__ void fwht_rows(float (*v)[kD], int g) {
  for (int s = 1; s < kD; s <<= 1) {
    for (int i = threadIdx.x; i < g * (kD / 2); i += kThreads) {
      const int h = i / (kD / 2), k = i % (kD / 2);
      const int lo = ((k & ~(s - 1)) << 1) | (k & (s - 1));
      const float a = v[h][lo], b = v[h][lo + s];
      v[h][lo] = a + b;
      v[h][lo + s] = a - b;
    }
    __syncthreads();
  }
  for (int i = threadIdx.x; i < g * kD; i += kThreads) v[i / kD][i % kD] *= kInvSqrt128;
  __syncthreads();
}

// grid: (nsplit, hkv, batch); block 128.
// FMT: the record format (RecFmt): yhat_td = alpha_t beta_d q_td + gamma_t delta_d.
template <int FMT>
__global__ void __launch_bounds__(kThreads) decode_simple_kernel(DecodeArgs a) {
  using F = RecFmt<FMT>;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  DecodeSmem& S = *reinterpret_cast<DecodeSmem*>(smem_raw);
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x;
  const int g = a.g;

  int len = a.seq_lens[b];
  if (len < 0 || len > a.max_seq || len / kT > a.max_blocks) {
    if (split == 0 && kvh == 0 && tid == 0) report(a.status, KVARN_STATUS_BAD_LENGTH);
    len = 0;
  }
  // pages are split in runs of pages_per_split; the split holding the last
  // page also takes the fp16 tail (one extra unit)
  const int nfull = len / kT, rem = len % kT;
  const int nsb = nfull > 0 ? (nfull + a.pages_per_split - 1) / a.pages_per_split : 1;
  if (split >= nsb) return;
  const int u0 = split * a.pages_per_split;
  const int u1 = min(nfull, u0 + a.pages_per_split) + ((split == nsb - 1 && rem > 0) ? 1 : 0);

  // queries of the group: raw and rotated
  const __half* qb = a.q + ((int64_t)b * a.hq + (int64_t)kvh * g) * kD;
  for (int i = tid; i < g * kD; i += kThreads) {
    const float x = __half2float(qb[i]);
    S.qraw[i / kD][i % kD] = x;
    S.qrot[i / kD][i % kD] = x;
  }
  if (tid < g) {
    S.m[tid] = -INFINITY;
    S.l[tid] = 0.f;
  }
  __syncthreads();
  fwht_rows(S.qrot, g);

  float acc[kMaxG], acc_tail[kMaxG];
#pragma unroll
  for (int h = 0; h < kMaxG; ++h) acc[h] = acc_tail[h] = 0.f;

  for (int u = u0; u < u1; ++u) {
    float sc[kMaxG];
    if (u < nfull) {
      const int64_t page = a.block_table[(int64_t)b * a.max_blocks + u];
      if (page < 0 || page >= a.num_pages) {
        if (tid == 0) report(a.status, KVARN_STATUS_BAD_PAGE);
        continue;
      }
      const uint4* src =
          reinterpret_cast<const uint4*>(a.pool + (page * a.hkv + kvh) * (int64_t)F::bytes);
      uint4* dst = reinterpret_cast<uint4*>(S.rec);
      for (int i = tid; i < F::bytes / 16; i += kThreads) dst[i] = __ldg(src + i);
      __syncthreads();
      // qc = H q * beta^K (thread = channel), and sum_d H q * delta^K per head
      {
        const float2 bd = F::get_bd(S.rec + F::kc, tid);
        float part[kMaxG], part1[kMaxG];
        for (int h = 0; h < g; ++h) {
          const float x = S.qrot[h][tid] * bd.x;
          S.qc[h][tid] = x;
          part[h] = F::pc ? S.qrot[h][tid] * bd.y : x;
          if (F::g64) {   // channel groups 0-63 and 64-127
            part1[h] = tid >= 64 ? part[h] : 0.f;
            part[h] = tid < 64 ? part[h] : 0.f;
          }
        }
        block_reduce<false>(S, part, g, S.sq);
        if (F::g64) block_reduce<false>(S, part1, g, S.sq1);
      }
      // scores (thread = token)
      {
        const uint32_t* row =
            reinterpret_cast<const uint32_t*>(S.rec + kOffKCodes + (F::k8 ? 128 : 64) * tid);
        const float2 sz = F::get_sz_g(S.rec + F::ksz, tid, 0);
        float sc1[kMaxG];
        for (int h = 0; h < g; ++h) sc[h] = sc1[h] = 0.f;
        if constexpr (F::k8) {
          // byte e of word w is channel (4w + e) ^ 16 (t & 1) (k8_byte)
          for (int w = 0; w < 32; ++w) {
            const uint32_t word = row[w];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float code = (float)((word >> (8 * e)) & 255u);
              const int d = (4 * w + e) ^ (16 * (tid & 1));
              for (int h = 0; h < g; ++h) sc[h] = fmaf(S.qc[h][d], code, sc[h]);
            }
          }
        } else {
          for (int w = 0; w < 16; ++w) {
            const uint32_t word = row[w];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float code = (float)((word >> (4 * e)) & 15u);
              const int d = 8 * w + e;
              if (F::g64 && w >= 8) {   // channels 64..127: the second group
                for (int h = 0; h < g; ++h) sc1[h] = fmaf(S.qc[h][d], code, sc1[h]);
              } else {
                for (int h = 0; h < g; ++h) sc[h] = fmaf(S.qc[h][d], code, sc[h]);
              }
            }
          }
        }
        if (F::g64) {
          const float2 sz1 = F::get_sz_g(S.rec + F::ksz, tid, 1);
          for (int h = 0; h < g; ++h)
            sc[h] = a.scale * (fmaf(sz.x, sc[h], sz.y * S.sq[h]) +
                               fmaf(sz1.x, sc1[h], sz1.y * S.sq1[h]));
        } else {
          for (int h = 0; h < g; ++h) sc[h] = a.scale * fmaf(sz.x, sc[h], sz.y * S.sq[h]);
        }
      }
    } else {
      // fp16 tail tokens 0..rem-1 (thread = token), plain space
      for (int h = 0; h < g; ++h) sc[h] = -INFINITY;
      if (tid < rem) {
        const __half* kt = a.tail_k + (((int64_t)b * a.hkv + kvh) * kT + tid) * kD;
        for (int h = 0; h < g; ++h) sc[h] = 0.f;
        for (int d = 0; d < kD; ++d) {
          const float kd = __half2float(kt[d]);
          for (int h = 0; h < g; ++h) sc[h] = fmaf(S.qraw[h][d], kd, sc[h]);
        }
        for (int h = 0; h < g; ++h) sc[h] *= a.scale;
      }
    }
    // online softmax update
    {
      float mx[kMaxG];
      for (int h = 0; h < g; ++h) mx[h] = sc[h];
      block_reduce<true>(S, mx, g, S.alpha);   // alpha <- page max (temporarily)
      if (tid < g) {
        const float mnew = fmaxf(S.m[tid], S.alpha[tid]);
        const float al = S.m[tid] == -INFINITY ? 0.f : __expf(S.m[tid] - mnew);
        S.m[tid] = mnew;
        S.alpha[tid] = al;
      }
      __syncthreads();
    }
    float p[kMaxG];
    for (int h = 0; h < g; ++h) p[h] = sc[h] == -INFINITY ? 0.f : __expf(sc[h] - S.m[h]);
    if (u < nfull) {
      const float2 szv = F::get_sz_g(S.rec + F::vsz, tid, 0);
      float zp[kMaxG];
      for (int h = 0; h < g; ++h) {
        S.pw[h][tid] = p[h] * szv.x;
        zp[h] = p[h] * szv.y;
      }
      block_reduce<false>(S, zp, g, S.zs);
      if (F::g64) {   // the second channel group's s', z'
        const float2 szv1 = F::get_sz_g(S.rec + F::vsz, tid, 1);
        for (int h = 0; h < g; ++h) {
          S.pw1[h][tid] = p[h] * szv1.x;
          zp[h] = p[h] * szv1.y;
        }
        block_reduce<false>(S, zp, g, S.zs1);
      }
      block_reduce<false>(S, p, g, S.sq);  // S.sq: the page's sum of p per head
      if (tid < g) S.l[tid] = S.l[tid] * S.alpha[tid] + S.sq[tid];
      __syncthreads();
      // value sum (thread = channel d), rotated space
      {
        const int d = tid;
        const uint32_t* vw = reinterpret_cast<const uint32_t*>(S.rec + F::kpart);
        const float2 bdv = F::get_bd(S.rec + F::vc, d);
        // the channel's group: its s'^V-weighted probabilities and z' sum
        const bool second = F::g64 && d >= 64;
        float (*pw)[kT] = second ? S.pw1 : S.pw;
        const float* zs = second ? S.zs1 : S.zs;
        float pv[kMaxG];
        for (int h = 0; h < g; ++h) pv[h] = 0.f;
        if constexpr (F::v4) {
          // 4-bit codes: words p of token digit j; nibble n = 4s + u holds token
          // 16 (2p + (u >> 1)) + 8 (u & 1) + 2j + s
          for (int w = 0; w < 16; ++w) {
            const int j = w >> 2, pp = w & 3;
            const uint32_t word = vw[v4_word(d, j, pp)];
#pragma unroll
            for (int n = 0; n < 8; ++n) {
              const float code = (float)((word >> (4 * n)) & 15u);
              const int u = n & 3;
              const int t = 16 * (2 * pp + (u >> 1)) + 8 * (u & 1) + 2 * j + (n >> 2);
              for (int h = 0; h < g; ++h) pv[h] = fmaf(pw[h][t], code, pv[h]);
            }
          }
        } else {
          for (int w = 0; w < 8; ++w) {
            const int j = w >> 1, hh = w & 1;
            const uint32_t word = vw[v_word(d, j, hh)];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float code = (float)((word >> (2 * e)) & 3u);
              const int t = v_token(j, hh, e);
              for (int h = 0; h < g; ++h) pv[h] = fmaf(pw[h][t], code, pv[h]);
            }
          }
        }
        for (int h = 0; h < g; ++h) {
          const float u = F::pc ? fmaf(bdv.x, pv[h], bdv.y * zs[h]) : bdv.x * (pv[h] + zs[h]);
          acc[h] = fmaf(acc[h], S.alpha[h], u);
          acc_tail[h] *= S.alpha[h];
        }
      }
    } else {
      for (int h = 0; h < g; ++h) S.pw[h][tid] = p[h];
      block_reduce<false>(S, p, g, S.sq);
      if (tid < g) S.l[tid] = S.l[tid] * S.alpha[tid] + S.sq[tid];
      __syncthreads();
      const int d = tid;
      const __half* vt = a.tail_v + ((int64_t)b * a.hkv + kvh) * kT * kD;
      float pv[kMaxG];
      for (int h = 0; h < g; ++h) pv[h] = 0.f;
      for (int t = 0; t < rem; ++t) {
        const float vd = __half2float(vt[(int64_t)t * kD + d]);
        for (int h = 0; h < g; ++h) pv[h] = fmaf(S.pw[h][t], vd, pv[h]);
      }
      for (int h = 0; h < g; ++h) {
        acc[h] *= S.alpha[h];
        acc_tail[h] = fmaf(acc_tail[h], S.alpha[h], pv[h]);
      }
    }
    __syncthreads();  // the record and pw are rewritten by the next unit
  }

  // back to plain space: o = H acc + acc_tail
  for (int h = 0; h < g; ++h) S.qc[h][tid] = acc[h];
  __syncthreads();
  fwht_rows(S.qc, g);
  float o[kMaxG];
  for (int h = 0; h < g; ++h) o[h] = S.qc[h][tid] + acc_tail[h];

  __half* ob = a.out + ((int64_t)b * a.hq + (int64_t)kvh * g) * kD;
  if (nsb == 1) {
    for (int h = 0; h < g; ++h) {
      const float l = S.l[h];
      ob[h * kD + tid] = __float2half_rn(l > 0.f ? o[h] / l : 0.f);
    }
    return;
  }
  // split-K: publish the partial state, the last CTA of (b, kvh) merges
  const int64_t stride_split = kPartStride;
  for (int h = 0; h < g; ++h) {
    float* P = a.ws_part + (((int64_t)b * a.hq + kvh * g + h) * a.nsplit + split) * stride_split;
    if (tid == 0) {
      P[0] = S.m[h];
      P[1] = S.l[h];
    }
    P[4 + tid] = o[h];
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) S.ticket = atomicAdd(a.ws_count + (int64_t)b * a.hkv + kvh, 1);
  __syncthreads();
  if (S.ticket != nsb - 1) return;
  __threadfence();
  for (int h = 0; h < g; ++h) {
    const float* P = a.ws_part + (((int64_t)b * a.hq + kvh * g + h) * a.nsplit) * stride_split;
    float M = -INFINITY;
    for (int s2 = 0; s2 < nsb; ++s2) M = fmaxf(M, __ldcg(P + s2 * stride_split));
    float L = 0.f, O = 0.f;
    for (int s2 = 0; s2 < nsb; ++s2) {
      const float ms = __ldcg(P + s2 * stride_split);
      if (ms == -INFINITY) continue;
      const float w = __expf(ms - M);
      L = fmaf(w, __ldcg(P + s2 * stride_split + 1), L);
      O = fmaf(w, __ldcg(P + s2 * stride_split + 4 + tid), O);
    }
    ob[h * kD + tid] = __float2half_rn(L > 0.f ? O / L : 0.f);
  }
  if (tid == 0) a.ws_count[(int64_t)b * a.hkv + kvh] = 0;
}

template <int FMT>
cudaError_t launch_simple(const DecodeArgs& a, cudaStream_t s) {
  static std::atomic<uint64_t> smem_set{0};
  const int smem = (int)sizeof(DecodeSmem);
  cudaError_t e = ensure_dynamic_smem(decode_simple_kernel<FMT>, smem, smem_set);
  if (e != cudaSuccess) return e;
  dim3 grid(a.nsplit, a.hkv, a.batch);
  decode_simple_kernel<FMT><<<grid, kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

static_assert(sizeof(DecodeSmem) <= 232448, "one CTA's shared memory is at most 227 KB");

// Resident CTAs per SM of the CUDA-core decode: its shared memory (228 KB
// per SM, 1 KB reserved per CTA), at most 4.  Host-only arithmetic.
int decode_simple_ctas_per_sm() {
  const int n = 233472 / ((int)sizeof(DecodeSmem) + 1024);
  return n < 4 ? n : 4;
}

cudaError_t launch_decode_simple(const DecodeArgs& a, cudaStream_t s) {
  if (a.fmt == kFmtM16) return launch_simple<kFmtM16>(a, s);
  if (a.fmt == kFmtPC) return launch_simple<kFmtPC>(a, s);
  if (a.fmt == kFmtG64) return launch_simple<kFmtG64>(a, s);
  if (a.fmt == kFmtV4) return launch_simple<kFmtV4>(a, s);
  if (a.fmt == kFmtK8) return launch_simple<kFmtK8>(a, s);
  return launch_simple<kFmtF32>(a, s);
}

}  // namespace kvarn
