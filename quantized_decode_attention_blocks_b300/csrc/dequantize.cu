// dequantize.cu -- diagnostic dequantization of page records back to the
// rotated space, the inverse of the packing of the KVarN page's stage
// "Kuantize Edilmis Onbellek" (blog.edumints.com, "KVarN Nasil Calisir?"),
// for every record format: yhat_td = alpha_t beta_d q_td + gamma_t delta_d.
// Not on the hot path.
#include "kvarn_internal.cuh"

namespace kvarn {
namespace {

// Code of channel d, token t of the K part (4-bit natural order, or the
// 8-bit byte map of format 5).
template <int FMT>
__device__ __forceinline__ int k_code(const uint8_t* rec, int d, int t) {
  if constexpr (RecFmt<FMT>::k8)
    return rec[k8_byte(d, t)];
  else
    return (rec[64 * t + d / 2] >> (4 * (d & 1))) & 15;
}

// Code of channel d, token t = 16k + 8f + 2j + s of the V part (its codes
// open the part): 2-bit crumb 2(k & 3) + f + 8s of word v_word(d, j, k >> 2),
// or 4-bit nibble 4s + 2(k & 1) + f of word v4_word(d, j, k >> 1).
template <int FMT>
__device__ __forceinline__ int v_code(const uint8_t* vpart, int d, int t) {
  const int k = t >> 4, f = (t >> 3) & 1, j = (t >> 1) & 3, s = t & 1;
  const uint32_t* w = reinterpret_cast<const uint32_t*>(vpart);
  if constexpr (RecFmt<FMT>::v4)
    return (w[v4_word(d, j, k >> 1)] >> (4 * (4 * s + 2 * (k & 1) + f))) & 15;
  else
    return (w[v_word(d, j, k >> 2)] >> (2 * (2 * (k & 3) + f + 8 * s))) & 3;
}

// grid: n records; block 128 (thread = token).  yk/yv[n][128][128], in the
// oracle's order of operations: c_d (s'_t q + z'_t), or r_t (cs_d q + cz_d).
template <int FMT>
__global__ void __launch_bounds__(128) dequantize_kernel(const uint8_t* recs, float* yk,
                                                         float* yv) {
  using F = RecFmt<FMT>;
  const uint8_t* rec = recs + (int64_t)blockIdx.x * F::bytes;
  const uint8_t* vpart = rec + F::kpart;
  const int t = threadIdx.x;
  float* ok = yk + ((int64_t)blockIdx.x * kT + t) * kD;
  float* ov = yv + ((int64_t)blockIdx.x * kT + t) * kD;
  for (int d = 0; d < kD; ++d) {
    const int grp = F::g64 ? d >> 6 : 0;
    const float2 azk = F::get_sz_g(rec + F::ksz, t, grp);
    const float2 azv = F::get_sz_g(rec + F::vsz, t, grp);
    const float2 bdk = F::get_bd(rec + F::kc, d);
    const float2 bdv = F::get_bd(rec + F::vc, d);
    const float qk = (float)k_code<FMT>(rec, d, t), qv = (float)v_code<FMT>(vpart, d, t);
    if constexpr (F::pc) {   // r_t (cs_d q + cz_d)
      ok[d] = azk.x * fmaf(bdk.x, qk, bdk.y);
      ov[d] = azv.x * fmaf(bdv.x, qv, bdv.y);
    } else {                 // c_d (s'_t q + z'_t)
      ok[d] = bdk.x * fmaf(azk.x, qk, azk.y);
      ov[d] = bdv.x * fmaf(azv.x, qv, azv.y);
    }
  }
}

template <int FMT>
cudaError_t launch_fmt(const uint8_t* rec, int64_t n, float* yk, float* yv, cudaStream_t s) {
  dequantize_kernel<FMT><<<(unsigned)n, 128, 0, s>>>(rec, yk, yv);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dequantize(int fmt, const uint8_t* rec, int64_t n, float* yk, float* yv,
                              cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  switch (fmt) {
    case kFmtM16: return launch_fmt<kFmtM16>(rec, n, yk, yv, s);
    case kFmtPC: return launch_fmt<kFmtPC>(rec, n, yk, yv, s);
    case kFmtG64: return launch_fmt<kFmtG64>(rec, n, yk, yv, s);
    case kFmtV4: return launch_fmt<kFmtV4>(rec, n, yk, yv, s);
    case kFmtK8: return launch_fmt<kFmtK8>(rec, n, yk, yv, s);
    default: return launch_fmt<kFmtF32>(rec, n, yk, yv, s);
  }
}

}  // namespace kvarn
