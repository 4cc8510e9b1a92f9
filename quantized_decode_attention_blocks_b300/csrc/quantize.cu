// quantize.cu -- KVarN-style block quantization of 128-token x 128-channel
// tiles: Hadamard rotation, Sinkhorn-like log-domain variance normalization,
// asymmetric RTN (K 4-bit, V 2-bit), packing into the page record.
//
// Source of the method: "KVarN: Huawei'den KV-Cache Kuantizasyonu icin Yerel
// vLLM Backend'i" (blog.edumints.com), section "KVarN Nasil Calisir?", stages
// "Dondurulmus Onbellek" (rotation), "Normalize Edilmis Onbellek"
// (normalization) and "Kuantize Edilmis Onbellek" (RTN); format kvarn_k4v2_g128.
//
// One CTA of 128 threads quantizes one tile.  Thread t owns token row t in
// registers for the rotation, the row steps of the normalization and the
// per-token RTN; the rotated tile is also kept in shared memory, padded to a
// stride of 129 floats, so that thread d can walk channel column d without
// bank conflicts for the column steps and the channel-major V packing.
//
// Arithmetic notes (all fp32):
//  * y_t = H x_t by a 7-stage in-register Walsh-Hadamard butterfly, then
//    scaled by 1/sqrt(128);
//  * the log-domain updates a_t += log std(Z_t), Z = Y exp(-a - b), reduce to
//    a_t = log std_d(Y_td exp(-b_d)) (the old a_t cancels), and likewise for
//    b_d, so the kernel keeps 1/r_t and c_d, 1/c_d directly;
//  * the stored row metadata never needs r_t: s' = r (max - min)/(2^b - 1) of
//    Y/(r c) equals (max - min)/(2^b - 1) of Y/c, and z' = min of Y/c; the
//    codes u = (x - min)/s are invariant to the row scale as well.
#include "kvarn_internal.cuh"

namespace kvarn {
namespace {

constexpr int kPitch = kD + 1;  // padded row pitch of the shared tile (floats)

__device__ __forceinline__ void load_row_f32(const __half* src, bool coherent, float (&y)[kD]) {
  const uint4* p = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int i = 0; i < kD / 8; ++i) {
    uint4 u = coherent ? __ldcg(p + i) : __ldg(p + i);
    const __half2* h2 = reinterpret_cast<const __half2*>(&u);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float2 f = __half22float2(h2[e]);
      y[8 * i + 2 * e] = f.x;
      y[8 * i + 2 * e + 1] = f.y;
    }
  }
}

// In-register Walsh-Hadamard transform, natural (Sylvester) order.
__device__ __forceinline__ void fwht128(float (&y)[kD]) {
#pragma unroll
  for (int h = 1; h < kD; h <<= 1) {
#pragma unroll
    for (int i = 0; i < kD; ++i) {
      if ((i & h) == 0) {
        float a = y[i], b = y[i + h];
        y[i] = a + b;
        y[i + h] = a - b;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kD; ++i) y[i] *= kInvSqrt128;
}

// Centred population variance of w_i = v_i * f_i (two passes) and its mean.
struct Moments {
  float mean, var;
};

__device__ __forceinline__ bool skip_step(const Moments& m) {
  // variance <= 1e-10 * mean square, with mean square = var + mean^2
  return !(m.var > 1e-10f * (m.var + m.mean * m.mean));
}

// Quantizes the tile whose token t starts at x + t*ld (fp16, 16-byte aligned)
// into the K (part 0) or V (part 1) half of the page record `rec`.
// Must be called by all 128 threads of the CTA; sY has kT*kPitch floats,
// svec has 5*kD floats.
__device__ void quantize_tile(const __half* x, int64_t ld, bool coherent, uint8_t* rec, int part,
                              int iters, float* sY, float* svec) {
  const int t = threadIdx.x;
  float* ra = svec;            // 1 / r_t
  float* cb = svec + kD;       // 1 / c_d
  float* cc = svec + 2 * kD;   // c_d
  float* zmin = svec + 3 * kD; // V packing: per-token min of Y/c
  float* sinv = svec + 4 * kD; // V packing: per-token (2^b - 1) / (max - min)

  float y[kD];
  load_row_f32(x + (int64_t)t * ld, coherent, y);
  fwht128(y);
#pragma unroll
  for (int d = 0; d < kD; ++d) sY[t * kPitch + d] = y[d];
  ra[t] = 1.f;
  cb[t] = 1.f;
  cc[t] = 1.f;
  __syncthreads();

  for (int it = 0; it < iters; ++it) {
    // row step: thread t, Z_t. = Y_t. * cb
    {
      float s = 0.f;
#pragma unroll
      for (int d = 0; d < kD; ++d) s = fmaf(y[d], cb[d], s);
      Moments m;
      m.mean = s * (1.f / kD);
      float v = 0.f;
#pragma unroll
      for (int d = 0; d < kD; ++d) {
        float e = fmaf(y[d], cb[d], -m.mean);
        v = fmaf(e, e, v);
      }
      m.var = v * (1.f / kD);
      if (!skip_step(m)) ra[t] = 1.f / sqrtf(m.var);
    }
    __syncthreads();
    // column step: thread d = t, Z_.d = Y_.d * ra
    {
      const int d = t;
      float s = 0.f;
      for (int r = 0; r < kT; ++r) s = fmaf(sY[r * kPitch + d], ra[r], s);
      Moments m;
      m.mean = s * (1.f / kT);
      float v = 0.f;
      for (int r = 0; r < kT; ++r) {
        float e = fmaf(sY[r * kPitch + d], ra[r], -m.mean);
        v = fmaf(e, e, v);
      }
      m.var = v * (1.f / kT);
      if (!skip_step(m)) {
        float c = sqrtf(m.var);
        cc[d] = c;
        cb[d] = 1.f / c;
      }
    }
    __syncthreads();
  }

  // per-token RTN on x'_td = Y_td / c_d
  const int qmax = part == 0 ? 15 : 3;
  float mn = INFINITY, mx = -INFINITY;
#pragma unroll
  for (int d = 0; d < kD; ++d) {
    y[d] *= cb[d];
    mn = fminf(mn, y[d]);
    mx = fmaxf(mx, y[d]);
  }
  const float range = mx - mn;
  const float s_out = range / (float)qmax;
  const float inv = range > 0.f ? (float)qmax / range : 0.f;
  {
    float2 meta = make_float2(s_out, mn);
    *reinterpret_cast<float2*>(rec + (part == 0 ? kOffKSZ : kOffVSZ) + 8 * t) = meta;
    reinterpret_cast<float*>(rec + (part == 0 ? kOffKC : kOffVC))[t] = cc[t];
  }
  if (part == 0) {
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      uint32_t acc = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        float u = (y[8 * i + e] - mn) * inv;
        int qv = __float2int_rn(u);
        qv = min(max(qv, 0), 15);
        acc |= (uint32_t)qv << (4 * e);
      }
      w[i] = acc;
    }
    uint4* dst = reinterpret_cast<uint4*>(rec + kOffKCodes + 64 * t);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
  } else {
    // publish per-token min and 1/s, then thread d packs channel column d
    zmin[t] = mn;
    sinv[t] = inv;
    __syncthreads();
    const int d = t;
    const float cbd = cb[d];
    uint32_t* vw = reinterpret_cast<uint32_t*>(rec + kOffVCodes);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t w[2];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t acc = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int r = v_token(j, hh, i);
          float xv = sY[r * kPitch + d] * cbd;
          float u = (xv - zmin[r]) * sinv[r];
          int qv = __float2int_rn(u);
          qv = min(max(qv, 0), 3);
          acc |= (uint32_t)qv << (2 * i);
        }
        w[hh] = acc;
      }
      *reinterpret_cast<uint2*>(vw + v_word(d, j, 0)) = make_uint2(w[0], w[1]);
    }
  }
}

constexpr int kQuantSmem = (kT * kPitch + 5 * kD) * sizeof(float);

// grid: (max_seq/128 + 1, 2*hkv, batch); block 128.
__global__ void __launch_bounds__(128) quantize_blocks_kernel(QuantizeArgs a) {
  extern __shared__ float smem[];
  const int b = blockIdx.z;
  const int h = blockIdx.y >> 1;
  const int part = blockIdx.y & 1;
  const int j = blockIdx.x;
  const int len = a.seq_lens[b];
  if (len < 0 || len > a.max_seq) {
    if (j == 0 && blockIdx.y == 0 && threadIdx.x == 0) report(a.status, KVARN_STATUS_BAD_LENGTH);
    return;
  }
  const int nfull = len / kT, rem = len % kT;
  const __half* src = (part ? a.v : a.k) + (int64_t)b * a.sb + (int64_t)h * a.sh;
  if (j < nfull) {
    if (j >= a.max_blocks) {
      if (threadIdx.x == 0) report(a.status, KVARN_STATUS_BAD_LENGTH);
      return;
    }
    const int64_t page = a.block_table[(int64_t)b * a.max_blocks + j];
    if (page < 0 || page >= a.num_pages) {
      if (threadIdx.x == 0) report(a.status, KVARN_STATUS_BAD_PAGE);
      return;
    }
    uint8_t* rec = a.pool + (page * a.hkv + h) * (int64_t)kRec;
    quantize_tile(src + (int64_t)j * kT * a.st, a.st, false, rec, part, a.iters, smem,
                  smem + kT * kPitch);
  } else if (j == nfull && rem > 0) {
    __half* tail = (part ? a.tail_v : a.tail_k) + ((int64_t)b * a.hkv + h) * kT * kD;
    for (int i = threadIdx.x; i < rem * (kD / 8); i += blockDim.x) {
      const int r = i / (kD / 8), c = i % (kD / 8);
      const uint4* s4 = reinterpret_cast<const uint4*>(src + ((int64_t)nfull * kT + r) * a.st);
      reinterpret_cast<uint4*>(tail + (int64_t)r * kD)[c] = __ldg(s4 + c);
    }
  }
}

// grid: (2*hkv, batch); block 128.
__global__ void __launch_bounds__(128) append_token_kernel(AppendArgs a) {
  extern __shared__ float smem[];
  const int b = blockIdx.y;
  const int h = blockIdx.x >> 1;
  const int part = blockIdx.x & 1;
  const int p = a.pos[b];
  if (p < 0) return;
  const int slot = p % kT;
  __half* tail = (part ? a.tail_v : a.tail_k) + ((int64_t)b * a.hkv + h) * kT * kD;
  const __half* src = (part ? a.v_new : a.k_new) + ((int64_t)b * a.hkv + h) * kD;
  if (threadIdx.x < kD / 8)
    reinterpret_cast<uint4*>(tail + (int64_t)slot * kD)[threadIdx.x] =
        __ldg(reinterpret_cast<const uint4*>(src) + threadIdx.x);
  if (slot != kT - 1) return;
  __syncthreads();
  const int blk = p / kT;
  if (blk >= a.max_blocks) {
    if (threadIdx.x == 0) report(a.status, KVARN_STATUS_BAD_LENGTH);
    return;
  }
  const int64_t page = a.block_table[(int64_t)b * a.max_blocks + blk];
  if (page < 0 || page >= a.num_pages) {
    if (threadIdx.x == 0) report(a.status, KVARN_STATUS_BAD_PAGE);
    return;
  }
  uint8_t* rec = a.pool + (page * a.hkv + h) * (int64_t)kRec;
  quantize_tile(tail, kD, true, rec, part, a.iters, smem, smem + kT * kPitch);
}

// grid: n records; block 128.  yk/yv[n][128][128] = c_d (s'_t q_td + z'_t).
__global__ void __launch_bounds__(128) dequantize_kernel(const uint8_t* recs, float* yk, float* yv) {
  const uint8_t* rec = recs + (int64_t)blockIdx.x * kRec;
  const int t = threadIdx.x;
  float* ok = yk + (int64_t)blockIdx.x * kT * kD;
  float* ov = yv + (int64_t)blockIdx.x * kT * kD;
  const float2 mk = reinterpret_cast<const float2*>(rec + kOffKSZ)[t];
  const float2 mv = reinterpret_cast<const float2*>(rec + kOffVSZ)[t];
  const float* ck = reinterpret_cast<const float*>(rec + kOffKC);
  const float* cv = reinterpret_cast<const float*>(rec + kOffVC);
  for (int d = 0; d < kD; ++d) {
    const int qk = (rec[kOffKCodes + 64 * t + d / 2] >> (4 * (d & 1))) & 15;
    const int kk = t >> 4, f = (t >> 3) & 1, j = (t >> 1) & 3, sb = t & 1;
    const uint32_t vw = reinterpret_cast<const uint32_t*>(rec + kOffVCodes)[v_word(d, j, kk >> 2)];
    const int qv = (vw >> (2 * (2 * (kk & 3) + f + 8 * sb))) & 3;
    ok[t * kD + d] = ck[d] * fmaf(mk.x, (float)qk, mk.y);
    ov[t * kD + d] = cv[d] * fmaf(mv.x, (float)qv, mv.y);
  }
}

}  // namespace

cudaError_t launch_quantize_blocks(const QuantizeArgs& a, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(quantize_blocks_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kQuantSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(append_token_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kQuantSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(a.max_seq / kT + 1, 2 * a.hkv, a.batch);
  quantize_blocks_kernel<<<grid, 128, kQuantSmem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_append_token(const AppendArgs& a, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(append_token_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kQuantSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(2 * a.hkv, a.batch);
  append_token_kernel<<<grid, 128, kQuantSmem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_dequantize(const uint8_t* rec, int64_t n, float* yk, float* yv,
                              cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  dequantize_kernel<<<(unsigned)n, 128, 0, s>>>(rec, yk, yv);
  return cudaGetLastError();
}

}  // namespace kvarn
