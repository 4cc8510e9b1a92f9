// dequantize.cu -- diagnostic dequantization of page records back to the
// rotated space: yhat_td = c_d (s'_t q_td + z'_t), the inverse of the packing
// of the KVarN page's stage "Kuantize Edilmis Onbellek" (blog.edumints.com,
// "KVarN Nasil Calisir?").  Not on the hot path.
#include "kvarn_internal.cuh"

namespace kvarn {
namespace {

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

cudaError_t launch_dequantize(const uint8_t* rec, int64_t n, float* yk, float* yv,
                              cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  dequantize_kernel<<<(unsigned)n, 128, 0, s>>>(rec, yk, yv);
  return cudaGetLastError();
}

}  // namespace kvarn
