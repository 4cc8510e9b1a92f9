// chunk_attention.cu -- attention of a chunk of new query tokens over the
// quantized paged cache (chunked prefill), on the fifth-generation tensor
// cores.
//
// Method: every query token attends causally to the cached tokens up to its
// own position ("KV Cache (Anahtar-Deger Onbellegi)", yapayzekasozluk.tr, "KV
// Cache Nasil Calisir?"), the cache being paged ("Paged Attention (vLLM)") and
// quantized per the KVarN page (blog.edumints.com, "KVarN Nasil Calisir?"):
// keys and values are stored rotated, y = H x, and the orthonormal rotation
// keeps scores, so with q~ = H q
//     s_it = q~_i . yhatK_t,   o_i = H (sum_t p_it yhatV_t) / sum_t p_it,
// yhat_td = c_d (s'_t q_td + z'_t) for a page token (r_t (cs_d q_td + cz_d)
// for per-channel groups; the {s', z'} of the channel's group for groups of
// 64); a token of the fp16 tail is rotated on the way in (yhat = H x).
//
// CTA = one tile of 128 query rows of one (sequence, KV head): row r holds
// query token i0 + r / g of head r mod g of the KV head's group.  It walks the
// cache blocks (pages, then the tail) that the tile's last token can see, in
// the structure of a streaming-softmax attention:
//   S   = Q~ K^T   tcgen05.mma, M = 128 rows, N = 128 tokens, K = 128 channels,
//                  as three products Qhi Khi + Qhi Klo + Qlo Khi (fp16 operands
//                  split hi + lo: one fp16 keeps 11 bits, too few for scores
//                  against keys with outlier channels), fp32 in TMEM;
//   P   = 2^(S - m) fp16, causal mask, running max m with a lazy rescale of O
//         (only when the max grows by more than 2^8, which fp16 P holds),
//         written to TMEM;
//   O  += P V^      tcgen05.mma with A = P from TMEM, N = 128 channels, K = 128
//                  tokens, as P Vhi + P Vlo, fp32 in TMEM.
// Roles: warps 0-3 build Q~ once and run the softmax (thread r = TMEM lane r =
// row r); between the two passes over a block's scores they also dequantize
// its values into the V^ (hi, lo) operands.  Warps 4-6 bring each page record
// in with one bulk copy (two buffers, one block ahead; for the records of more
// than 15360 bytes one buffer, whose K part they load and whose V part the
// softmax warps load, each as soon as its part of the record before is read)
// and dequantize its keys into the K^ (hi, lo) operands (the fp16 tail is
// rotated on the way in).  One
// thread of warp 7 issues the MMAs, polling for whichever of the next S (one
// block ahead, two S buffers in TMEM) or the next PV has its inputs ready, so
// the tensor cores work on the next block's scores while the softmax warps
// work on this block's.  The hand-offs are mbarriers, every wait bounded
// (KVARN_STATUS_TIMEOUT).  At the end each softmax thread reads its row of O,
// divides by l, rotates it back with a register FWHT and writes fp16.
#include "kvarn_internal.cuh"
#include "ptx.cuh"

namespace kvarn {
namespace {

using namespace ptx;

constexpr int kSoftWarps = 4;                         // rows: TMEM lane quarters
constexpr int kDeqWarps = 3;                          // 8 warps in all: 255 registers
constexpr int kCThreads = 32 * (kSoftWarps + kDeqWarps + 1);
constexpr int kDeq0 = 32 * kSoftWarps;                // first dequant thread
constexpr int kMmaThread = 32 * (kSoftWarps + kDeqWarps);
constexpr uint32_t kOp = 128 * 128 * 2;               // one fp16 operand, 128 x 128
constexpr uint32_t kOpBox = kOp / 2;                  // 64-element-wide half
// TMEM columns: S (two buffers) [0, 256), O [256, 384), P (fp16 pairs) [384, 448)
constexpr uint32_t kCTmemCols = 512;
constexpr uint32_t kColO = 256, kColP = 384;
constexpr uint64_t kCWaitNs = 2000000000ull;
// kind::f16, fp16 A and B (both K-major), fp32 D, M = 128, N = 128
constexpr uint32_t kCIdesc = (1u << 4) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
constexpr float kLazy = 8.f;                          // log2 units

// RB: the record format's bytes; NRAW: page records in flight (two where
// they fit beside the six operands, else one).
template <int RB, int NRAW>
struct __align__(1024) CSmem {
  uint8_t qh[kOp];        // A of S: q~ high part   [row][channel]
  uint8_t ql[kOp];        //         q~ low part
  uint8_t kh[kOp];        // B of S: yhatK high     [token][channel]
  uint8_t kl[kOp];        //         yhatK low
  uint8_t vh[kOp];        // B of PV: yhatV high    [channel][token]
  uint8_t vl[kOp];        //          yhatV low
  uint8_t raw[NRAW][RB];  // page records in flight
  uint64_t raw_full[2];   // per buffer; with one buffer: [0] its K part, [1] its V part
  uint64_t sdone[2];      // S of a block ready, per S buffer
  uint64_t rawfree[2];    // a buffer's keys and values (one buffer: its keys; its values)
                          // are dequantized
  uint64_t qready, kready, vready, pready, pvdone, drain;
  uint32_t tmem_base;
  int abort;
};
// records in flight for a format: two for the 15360-byte (and smaller)
// records, one for the records of groups of 64, 4-bit values or 8-bit keys
template <int FMT>
constexpr int raw_buffers() {
  return (int)sizeof(CSmem<RecFmt<FMT>::bytes, 2>) + 1024 <= 232448 ? 2 : 1;
}
template <int FMT>
constexpr int chunk_smem_bytes() {
  return (int)sizeof(CSmem<RecFmt<FMT>::bytes, raw_buffers<FMT>()>) + 1024;
}
static_assert(raw_buffers<kFmtF32>() == 2 && raw_buffers<kFmtM16>() == 2 &&
                  raw_buffers<kFmtPC>() == 2 && raw_buffers<kFmtG64>() == 1 &&
                  raw_buffers<kFmtV4>() == 1 && raw_buffers<kFmtK8>() == 1,
              "the large records are single-buffered");
static_assert(chunk_smem_bytes<kFmtF32>() <= 232448 && chunk_smem_bytes<kFmtK8>() <= 232448 &&
                  chunk_smem_bytes<kFmtG64>() <= 232448 && chunk_smem_bytes<kFmtV4>() <= 232448,
              "shared memory of one CTA");

// Byte offset of the 16-byte chunk holding elements 8c .. 8c + 7 (c < 16) of
// row r of a 128 x 128 fp16 operand in the 128-byte swizzled K-major layout:
// two 64-element halves of 16 KB, rows of 128 bytes, chunk c & 7 of row r at
// position (c & 7) ^ (r & 7).
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
  return (uint32_t)((c >> 3) * kOpBox + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ float ex2c(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// In-place Walsh-Hadamard butterflies over 128 values in natural (Sylvester)
// order, unnormalised: x <- Hs x.
__device__ __forceinline__ void fwht128(float (&x)[128]) {
#pragma unroll
  for (int h = 1; h < 128; h <<= 1)
#pragma unroll
    for (int i = 0; i < 128; ++i)
      if ((i & h) == 0) {
        const float a = x[i], b = x[i + h];
        x[i] = a + b;
        x[i + h] = a - b;
      }
}

__device__ __forceinline__ void load_row(const __half* src, float (&x)[128]) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const uint4 u = __ldg(s4 + c);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
      x[8 * c + 2 * e] = f.x;
      x[8 * c + 2 * e + 1] = f.y;
    }
  }
}

__device__ __forceinline__ uint32_t h2bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// The fp16 pair (hi, lo) of two fp32 values: hi = fp16(x), lo = fp16(x - hi).
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 hf = __half22float2(h);
  hi = h2bits(h);
  lo = h2bits(__floats2half2_rn(a - hf.x, b - hf.y));
}

// 8 values of row r, chunk c, written as hi and lo parts
__device__ __forceinline__ void store_hilo8(uint8_t* hi, uint8_t* lo, int r, int c,
                                            const float* y) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) split2(y[2 * e], y[2 * e + 1], h[e], l[e]);
  const uint32_t o = sw_off(r, c);
  *reinterpret_cast<uint4*>(hi + o) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4*>(lo + o) = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ float code_f(uint32_t q) {   // small integer -> float, exact
  return __int_as_float(0x4B000000 | q) - 8388608.f;
}

// Page tokens: yhatK_td = c_d (s'_t q_td + z'_t) into the K^ operands.  Lane:
// chunk cc = lane & 15 (channels 8 cc .. 8 cc + 7, code word cc of a token
// row), t0 = lane >> 4; dequant warp dw takes the token pairs p = dw, dw + 3,
// ... of 64, token 2p + t0.  The code loads hit 32 banks, the column scales
// of the lane's chunk are loaded once.  rk: the record's K part.
template <int FMT>
__device__ __forceinline__ void dequant_k(const uint8_t* rk, uint8_t* kh, uint8_t* kl, int dw,
                                          int lane) {
  using F = RecFmt<FMT>;
  const int cc = lane & 15, t0 = lane >> 4;
  // beta (c, or cs for the per-channel format) and delta (c, or cz) of the
  // lane's 8 channels
  const float4 ca = F::get_b4(rk + F::kc, 2 * cc);
  const float4 cb = F::get_b4(rk + F::kc, 2 * cc + 1);
  const float cs[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
  float cz[8];
  if constexpr (F::pc) {
    const float4 za = F::get_d4(rk + F::kc, 2 * cc);
    const float4 zb = F::get_d4(rk + F::kc, 2 * cc + 1);
    cz[0] = za.x; cz[1] = za.y; cz[2] = za.z; cz[3] = za.w;
    cz[4] = zb.x; cz[5] = zb.y; cz[6] = zb.z; cz[7] = zb.w;
  }
  // four token pairs per step: independent loads and math in flight
  constexpr int kStep = 4 * kDeqWarps;
#pragma unroll 1
  for (int p0 = dw; p0 < kT / 2; p0 += kStep) {
    uint32_t w[4], w2[4];   // the 8 codes: nibbles of w, or bytes of w, w2 (8-bit keys)
    float2 sz[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int t = 2 * min(p0 + kDeqWarps * u, kT / 2 - 1) + t0;
      if constexpr (F::k8) {   // channels 8 cc .. of token t: 8 bytes at k8_byte(8 cc, t)
        const uint2 b8 = *reinterpret_cast<const uint2*>(rk + k8_byte(8 * cc, t));
        w[u] = b8.x;
        w2[u] = b8.y;
      } else {
        w[u] = *reinterpret_cast<const uint32_t*>(rk + kOffKCodes + 64 * t + 4 * cc);
        w2[u] = 0u;
      }
      sz[u] = F::get_sz_g(rk + F::ksz, t, F::g64 ? cc >> 3 : 0);   // the chunk's group
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int p = p0 + kDeqWarps * u;
      if (p >= kT / 2) break;
      float y[8];
#pragma unroll
      for (int k = 0; k < 8; k += 2) {
        float2 q2;
        if constexpr (F::k8) {
          const uint32_t wk = k < 4 ? w[u] : w2[u];
          q2 = make_float2(code_f((wk >> (8 * (k & 3))) & 255u),
                           code_f((wk >> (8 * (k & 3) + 8)) & 255u));
        } else {
          q2 = make_float2(code_f((w[u] >> (4 * k)) & 15u), code_f((w[u] >> (4 * k + 4)) & 15u));
        }
        float2 v;
        if constexpr (F::pc)   // r_t (cs_d q + cz_d)
          v = __fmul2_rn(make_float2(sz[u].x, sz[u].x),
                         __ffma2_rn(make_float2(cs[k], cs[k + 1]), q2,
                                    make_float2(cz[k], cz[k + 1])));
        else                   // c_d (s'_t q + z'_t)
          v = __fmul2_rn(make_float2(cs[k], cs[k + 1]),
                         __ffma2_rn(make_float2(sz[u].x, sz[u].x), q2,
                                    make_float2(sz[u].y, sz[u].y)));
        y[k] = v.x;
        y[k + 1] = v.y;
      }
      store_hilo8(kh, kl, 2 * p + t0, cc, y);
    }
  }
}

// Page tokens: yhatV into the V^ operands [channel][token].  Lane: j = lane &
// 3, r = lane >> 2; for each h (0, 1) warp dw of NW takes the rounds k2 =
// dw, dw + NW, ... of 16, m = k2 >> 1, e = k2 & 1, and reads word
// 128m + 16r + 4j + 2e + h of the permuted V code layout: channel
// c = 16m + 8e + r, tokens 16k + 8f + 2j + s for k = 4h .. 4h + 3.  The lanes
// of one store differ in (r, j), i.e. in 32 banks.
template <int NW, int FMT>
__device__ __forceinline__ void dequant_v(const uint8_t* rv, uint8_t* vh, uint8_t* vl, int dw,
                                          int lane) {
  using F = RecFmt<FMT>;
  const int j2 = lane & 3, r = lane >> 2;
  const uint8_t* vsz = rv + (F::vsz - F::kpart);
  const uint32_t* words = reinterpret_cast<const uint32_t*>(rv);   // V codes open the V part
  const uint8_t* vc = rv + (F::vc - F::kpart);
  if constexpr (F::v4) {
    // 4-bit codes: words p = 0..3 of (channel, j), nibble 4s + 2(k & 1) + f
    // of word p holding token 16k + 8f + 2j + s for k = 2p, 2p + 1
#pragma unroll 1
    for (int p = 0; p < 4; ++p) {
      float2 sz[2][2][2];
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)
#pragma unroll
        for (int f = 0; f < 2; ++f)
#pragma unroll
          for (int s = 0; s < 2; ++s)
            sz[kk][f][s] = F::get_sz(vsz, 16 * (2 * p + kk) + 8 * f + 2 * j2 + s);
#pragma unroll 2
      for (int k2 = dw; k2 < 16; k2 += NW) {
        const int m = k2 >> 1, e = k2 & 1;
        const int c = 16 * m + 8 * e + r;
        const uint32_t w = words[v4_word(c, j2, p)];
        const float cd = F::get_bd(vc, c).x;
#pragma unroll
        for (int kk = 0; kk < 2; ++kk)
#pragma unroll
          for (int f = 0; f < 2; ++f) {
            const int i0 = 2 * kk + f;   // nibble of s = 0; s = 1 is nibble i0 + 4
            const float q0 = code_f((w >> (4 * i0)) & 15u), q1 = code_f((w >> (4 * i0 + 16)) & 15u);
            const float y0 = cd * fmaf(sz[kk][f][0].x, q0, sz[kk][f][0].y);
            const float y1 = cd * fmaf(sz[kk][f][1].x, q1, sz[kk][f][1].y);
            const int u = 2 * (2 * p + kk) + f;   // tokens 8u .. 8u + 7
            const uint32_t off =
                (uint32_t)((u >> 3) * kOpBox + c * 128 + (((u & 7) ^ (c & 7)) << 4) + 4 * j2);
            uint32_t hi, lo;
            split2(y0, y1, hi, lo);
            *reinterpret_cast<uint32_t*>(vh + off) = hi;
            *reinterpret_cast<uint32_t*>(vl + off) = lo;
          }
      }
    }
  } else {
#pragma unroll 1
  for (int hb = 0; hb < 2; ++hb) {
    // the tokens' {s', z'} (of group 0 for groups of 64: group 1 is read
    // per channel below)
    float2 sz[4][2][2];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
      for (int f = 0; f < 2; ++f)
#pragma unroll
        for (int s = 0; s < 2; ++s)
          sz[kk][f][s] = F::get_sz_g(vsz, 16 * (4 * hb + kk) + 8 * f + 2 * j2 + s, 0);
#pragma unroll 2
    for (int k2 = dw; k2 < 16; k2 += NW) {
      const int m = k2 >> 1, e = k2 & 1;
      const int c = 16 * m + 8 * e + r;
      const uint32_t w = words[128 * m + 16 * r + 4 * j2 + 2 * e + hb];
      const float2 bd = F::get_bd(vc, c);   // (c, c), or (cs, cz) per channel
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int f = 0; f < 2; ++f) {
          const int i0 = 2 * kk + f;   // crumb of s = 0; s = 1 is crumb i0 + 8
          const float q0 = code_f((w >> (2 * i0)) & 3u), q1 = code_f((w >> (2 * i0 + 16)) & 3u);
          float2 sz0 = sz[kk][f][0], sz1 = sz[kk][f][1];
          if (F::g64 && c >= 64) {   // the second channel group's {s', z'}
            const int tok = 16 * (4 * hb + kk) + 8 * f + 2 * j2;
            sz0 = F::get_sz_g(vsz, tok, 1);
            sz1 = F::get_sz_g(vsz, tok + 1, 1);
          }
          float y0, y1;
          if constexpr (F::pc) {   // r_t (cs_d q + cz_d)
            y0 = sz0.x * fmaf(bd.x, q0, bd.y);
            y1 = sz1.x * fmaf(bd.x, q1, bd.y);
          } else {                 // c_d (s'_t q + z'_t)
            y0 = bd.x * fmaf(sz0.x, q0, sz0.y);
            y1 = bd.x * fmaf(sz1.x, q1, sz1.y);
          }
          const int u = 2 * (4 * hb + kk) + f;   // tokens 8u .. 8u + 7; these are 2 j2, 2 j2 + 1
          const uint32_t off =
              (uint32_t)((u >> 3) * kOpBox + c * 128 + (((u & 7) ^ (c & 7)) << 4) + 4 * j2);
          uint32_t hi, lo;
          split2(y0, y1, hi, lo);
          *reinterpret_cast<uint32_t*>(vh + off) = hi;
          *reinterpret_cast<uint32_t*>(vl + off) = lo;
        }
    }
  }
  }   // 2-bit codes
}

// FMT: the record format (RecFmt).
template <int FMT>
__global__ void __launch_bounds__(kCThreads, 1)
    chunk_attention_kernel(const ChunkArgs a) {
  using F = RecFmt<FMT>;
  constexpr int NRAW = raw_buffers<FMT>();
  using Smem = CSmem<F::bytes, NRAW>;
  extern __shared__ uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~static_cast<uintptr_t>(1023));
  // record buffer of block j and the parity of its use
  auto rb = [](int j) { return NRAW == 2 ? j & 1 : 0; };
  auto rph = [](int j) { return (uint32_t)((NRAW == 2 ? j >> 1 : j) & 1); };
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.z, kvh = blockIdx.y;
  const int tile = a.ntq - 1 - (int)blockIdx.x;   // longest tiles first
  const int g = a.g, tq = a.tq;
  const int i0 = tile * tq;
  const int start = a.start[b];
  int cl = a.chunk_lens[b];
  const int64_t n64 = (int64_t)start + cl;
  const bool bad =
      start < 0 || cl < 0 || cl > a.M || n64 > a.max_seq || n64 / kT > a.max_blocks;
  const int n = bad ? 0 : (int)n64;
  if (bad) {
    if (tile == 0 && kvh == 0 && tid == 0) report(a.status, KVARN_STATUS_BAD_LENGTH);
    cl = 0;
  }
  const int nfull = bad ? 0 : n / kT;
  const int last = min(i0 + tq, cl) - 1;           // last query token of the tile
  const int nblk = last >= 0 ? (start + last) / kT + 1 : 0;
  const int32_t* trow = a.block_table + (int64_t)b * a.max_blocks;
  // every page the tile reads must be in the pool
  int pbad = 0;
  for (int j = tid; j < min(nblk, nfull); j += kCThreads) {
    const int p = trow[j];
    if (p < 0 || (int64_t)p >= a.num_pages) pbad = 1;
  }
  if (__syncthreads_or(pbad)) {
    if (tid == 0) report(a.status, KVARN_STATUS_BAD_PAGE);
    cl = 0;
  }
  __half* const orow0 = a.out + (int64_t)b * a.M * a.hq * kD;
  if (cl <= i0) {
    // no query token of this tile: its rows (tokens below M) are zeros
    for (int x = tid; x < 128 * 16; x += kCThreads) {
      const int r = x >> 4, c = x & 15, i = i0 + r / g;
      if (r < tq * g && i < a.M)
        reinterpret_cast<uint4*>(orow0 + ((int64_t)i * a.hq + kvh * g + r % g) * kD)[c] =
            make_uint4(0u, 0u, 0u, 0u);
    }
    return;
  }

  if (tid == 0) {
    for (int x = 0; x < 2; ++x) {
      mbar_init(&S.raw_full[x], 1);
      // two buffers: both kinds of warps free a record; one buffer: the
      // dequant warps free its K part, the softmax warps its V part
      mbar_init(&S.rawfree[x], NRAW == 2 ? kSoftWarps + kDeqWarps : x == 0 ? kDeqWarps : kSoftWarps);
    }
    mbar_init(&S.qready, kSoftWarps);
    mbar_init(&S.kready, kDeqWarps);
    mbar_init(&S.vready, kSoftWarps);
    mbar_init(&S.sdone[0], 1);
    mbar_init(&S.sdone[1], 1);
    mbar_init(&S.pready, kSoftWarps);
    mbar_init(&S.pvdone, 1);
    mbar_init(&S.drain, 1);
    S.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&S.tmem_base, kCTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  auto wait = [&](uint64_t* bar, uint32_t ph) {
    if (*reinterpret_cast<volatile int*>(&S.abort)) return;
    if (!mbar_wait_bounded(bar, ph, kCWaitNs)) {
      *reinterpret_cast<volatile int*>(&S.abort) = 1;
      report(a.status, KVARN_STATUS_TIMEOUT);
    }
  };
  const int rem = n - nfull * kT;
  auto rec_of = [&](int j) {
    return a.pool + ((int64_t)trow[j] * a.hkv + kvh) * (int64_t)F::bytes;
  };
  const int npages = min(nblk, nfull);
  // one record buffer: its K and V parts stream separately, the dequant
  // warps loading the next K part and the softmax warps the next V part as
  // soon as their own part of the current record is dequantized
  auto issue_v = [&](int j) {
    mbar_arrive_expect_tx(&S.raw_full[1], F::vpart);
    bulk_g2s(S.raw[0] + F::kpart, rec_of(j) + F::kpart, F::vpart, &S.raw_full[1]);
  };

  if (warp < kSoftWarps) {
    // ================= softmax warps: row r = TMEM lane r =================
    const int r = tid, i = i0 + r / g, hh = r % g;
    uint32_t vissued = 0, vseen = 0;   // one buffer: V parts loaded / seen by tid 0
    const bool valid = r < tq * g && i < cl;
    const int Pr = valid ? start + i : -1;         // last key position of the row
    {
      float x[128];
      if (valid) {
        load_row(a.q + (((int64_t)b * a.M + i) * a.hq + kvh * g + hh) * kD, x);
        fwht128(x);
        const float f = kInvSqrt128 * a.scale_log2;   // scores in log2 units
#pragma unroll
        for (int d = 0; d < 128; ++d) x[d] *= f;
      } else {
#pragma unroll
        for (int d = 0; d < 128; ++d) x[d] = 0.f;
      }
#pragma unroll
      for (int c = 0; c < 16; ++c) store_hilo8(S.qh, S.ql, r, c, x + 8 * c);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.qready);

    const uint32_t tl = tmem + ((uint32_t)(32 * warp) << 16), tO = tl + kColO, tP = tl + kColP;
    const __half* tvb = a.tail_v + ((int64_t)b * a.hkv + kvh) * kT * kD;
    float m_ref = -INFINITY, l = 0.f;
    for (int j = 0; j < nblk; ++j) {
      const bool page = j < nfull;
      // S of block j is in buffer j & 1; two passes over it in 32-column pieces
      // (the maximum, then the probabilities), so no row sits in registers
      wait(&S.sdone[j & 1], (j >> 1) & 1);
      tc_fence_after();
      const uint32_t tS = tl + 128 * (j & 1);
      const int lim = Pr - kT * j;                  // columns 0 .. lim are visible
      float mb = -INFINITY;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        float sv[32];
        tmem_ld32(tS + 32 * c4, sv);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (32 * c4 + k <= lim) mb = fmaxf(mb, sv[k]);
      }
      // lazy rescale: a row moves its reference only when its maximum grows by
      // more than 2^kLazy; O holding earlier blocks is then rescaled.  The
      // TMEM accesses are warp-wide, so the warp rescales when any lane must
      // (alpha = 1 on the others)
      const bool grow = mb > m_ref + kLazy;
      const bool resc = grow && m_ref != -INFINITY;
      float alpha = 1.f;
      if (resc) {
        alpha = ex2c(m_ref - mb);
        l *= alpha;
      }
      if (grow) m_ref = mb;
      // PV of the block before is done: O is stable, V^ and P are free
      if (j > 0) wait(&S.pvdone, (j - 1) & 1);
      tc_fence_after();
      if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          float o[32];
          tmem_ld32(tO + 32 * c4, o);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] *= alpha;
          tmem_st32(tO + 32 * c4, o);
        }
        tmem_wait_st();
      }
      // ---- this block's values into V^ ----
      if (page) {
        if constexpr (NRAW == 2) {
          wait(&S.raw_full[rb(j)], rph(j));
        } else {
          wait(&S.raw_full[1], j & 1);
          if (tid == 0 && !*reinterpret_cast<volatile int*>(&S.abort)) ++vseen;
        }
        dequant_v<kSoftWarps, FMT>(S.raw[rb(j)] + F::kpart, S.vh, S.vl, warp, lane);
      } else {
        // the fp16 tail, rotated: column t = tid of V^ [channel][token]
        const int t = tid;
        float x[128];
        if (t < rem) {
          load_row(tvb + (int64_t)t * kD, x);
          fwht128(x);
#pragma unroll
          for (int d = 0; d < 128; ++d) x[d] *= kInvSqrt128;
        } else {
#pragma unroll
          for (int d = 0; d < 128; ++d) x[d] = 0.f;
        }
        const uint32_t tb = (uint32_t)((t >> 6) * kOpBox + (t & 7) * 2);
        const int tc = (t & 63) >> 3;
#pragma unroll
        for (int d = 0; d < 128; ++d) {
          const __half h = __float2half_rn(x[d]);
          const uint32_t o = tb + d * 128 + ((tc ^ (d & 7)) << 4);
          *reinterpret_cast<__half*>(S.vh + o) = h;
          *reinterpret_cast<__half*>(S.vl + o) = __float2half_rn(x[d] - __half2float(h));
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&S.vready);
        if (page) mbar_arrive(&S.rawfree[NRAW == 2 ? rb(j) : 1]);
      }
      if (NRAW == 1 && page && tid == 0 && j + 1 < npages &&
          !*reinterpret_cast<volatile int*>(&S.abort)) {
        wait(&S.rawfree[1], j & 1);   // every softmax warp read this V part
        issue_v(j + 1);
        ++vissued;
      }
      // ---- pass 2: P = 2^(S - m) as fp16 pairs into TMEM ----
      const bool any = m_ref != -INFINITY;
      float ls = 0.f;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        // columns 64 hf .. 64 hf + 63 of S -> fp16 pairs in P columns 32 hf ..
        float sv[64];
        tmem_ld32(tS + 64 * hf, sv);
        tmem_ld32(tS + 64 * hf + 32, sv + 32);
        tmem_wait_ld();
        float pw[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int c0 = 64 * hf + 2 * k;
          const float p0 = any && c0 <= lim ? ex2c(sv[2 * k] - m_ref) : 0.f;
          const float p1 = any && c0 + 1 <= lim ? ex2c(sv[2 * k + 1] - m_ref) : 0.f;
          const __half2 ph = __floats2half2_rn(p0, p1);
          const float2 pf = __half22float2(ph);     // l sums what the MMA multiplies
          ls += pf.x + pf.y;
          pw[k] = __uint_as_float(h2bits(ph));
        }
        tmem_st32(tP + 32 * hf, pw);
      }
      tmem_wait_st();
      l += ls;
      tc_fence_before();
      __syncwarp();
      // P is written and S buffer j & 1 is read
      if (lane == 0) mbar_arrive(&S.pready);
    }
    // ---- epilogue: o = H (O / l) / sqrt(128), fp16 ----
    wait(&S.pvdone, (nblk - 1) & 1);
    tc_fence_after();
    float o[128];
    tmem_ld32(tO, o);
    tmem_ld32(tO + 32, o + 32);
    tmem_ld32(tO + 64, o + 64);
    tmem_ld32(tO + 96, o + 96);
    tmem_wait_ld();
    if (r < tq * g && i < a.M) {
      uint4* dst = reinterpret_cast<uint4*>(orow0 + ((int64_t)i * a.hq + kvh * g + hh) * kD);
      if (valid && l > 0.f) {
        fwht128(o);
        const float f = kInvSqrt128 / l;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = h2bits(__floats2half2_rn(o[8 * c + 2 * e] * f, o[8 * c + 2 * e + 1] * f));
          dst[c] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    if (NRAW == 1 && tid == 0) {
      // V parts still in flight (a wait gave up) land before the CTA leaves:
      // the first was issued by the dequant warps, the others here
      const uint32_t total = (npages > 0 ? 1u : 0u) + vissued;
      for (uint32_t k = vseen; k < total; ++k) mbar_wait_bounded(&S.raw_full[1], k & 1, kCWaitNs);
    }
  } else if (warp < kSoftWarps + kDeqWarps) {
    // ================= dequant warps: page records in, keys into K^ =================
    const int dt = tid - kDeq0, dw = dt >> 5;
    // loads issued and seen complete per buffer (thread dt == 0), as
    // count0 | count1 << 16 so that no array sits in local memory
    uint32_t issued = 0, seen = 0;
    // the record of block j (two buffers), or its K part (one buffer)
    auto issue = [&](int j) {
      constexpr uint32_t bytes = NRAW == 2 ? F::bytes : F::kpart;
      uint64_t* bar = &S.raw_full[rb(j)];
      mbar_arrive_expect_tx(bar, bytes);
      bulk_g2s(S.raw[rb(j)], rec_of(j), bytes, bar);
      issued += 1u << (16 * rb(j));
    };
    if (dt == 0) {
      if (0 < npages) issue(0);
      if (NRAW == 2 && 1 < npages) issue(1);
      if (NRAW == 1 && 0 < npages) issue_v(0);
    }
    const __half* tkb = a.tail_k + ((int64_t)b * a.hkv + kvh) * kT * kD;
    for (int j = 0; j < nblk; ++j) {
      const bool page = j < nfull;
      if (page) {
        wait(&S.raw_full[rb(j)], rph(j));
        if (dt == 0 && !*reinterpret_cast<volatile int*>(&S.abort)) seen += 1u << (16 * rb(j));
      }
      if (j > 0) wait(&S.sdone[(j - 1) & 1], ((j - 1) >> 1) & 1);   // S of block j-1 read K^
      if (page) {
        dequant_k<FMT>(S.raw[rb(j)], S.kh, S.kl, dw, lane);
      } else {
        // the fp16 tail, rotated into the pages' space: yhat = H x / sqrt(128)
#pragma unroll 1
        for (int t = dt; t < kT; t += 32 * kDeqWarps) {
          float x[128];
          if (t < rem) {
            load_row(tkb + (int64_t)t * kD, x);
            fwht128(x);
#pragma unroll
            for (int d = 0; d < 128; ++d) x[d] *= kInvSqrt128;
          } else {
#pragma unroll
            for (int d = 0; d < 128; ++d) x[d] = 0.f;
          }
#pragma unroll
          for (int c = 0; c < 16; ++c) store_hilo8(S.kh, S.kl, t, c, x + 8 * c);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&S.kready);
        if (page) mbar_arrive(&S.rawfree[rb(j)]);
      }
      // two buffers: the buffer of block j - 1 is free once its values are
      // dequantized too, load block j + 1 into it; one buffer: the K part
      // of block j is free once every dequant warp read it, load the next K
      // part into it
      if (dt == 0 && j + 1 >= NRAW && j + 1 < npages &&
          !*reinterpret_cast<volatile int*>(&S.abort)) {
        wait(&S.rawfree[rb(j + 1 - NRAW)], rph(j + 1 - NRAW));
        issue(j + 1);
      }
    }
    if (dt == 0) {
      // copies still in flight (a wait gave up) land before the CTA leaves
#pragma unroll
      for (int s2 = 0; s2 < NRAW; ++s2)
        for (int k = (int)((seen >> (16 * s2)) & 0xFFFF); k < (int)((issued >> (16 * s2)) & 0xFFFF);
             ++k)
          mbar_wait_bounded(&S.raw_full[s2], (uint32_t)(k & 1), kCWaitNs);
    }
  } else if (tid == kMmaThread) {
    // ================= MMA issue =================
    // S_js (one block ahead, into S buffer js & 1, whose softmax of block
    // js - 2 is done) and PV_jp are issued as soon as their inputs are ready,
    // polled in turn, so neither waits for the other's inputs
    const uint32_t tO = tmem + kColO, tP = tmem + kColP;
    const uint32_t qh = smem_u32(S.qh), ql = smem_u32(S.ql), kh = smem_u32(S.kh),
                   kl = smem_u32(S.kl), vh = smem_u32(S.vh), vl = smem_u32(S.vl);
    wait(&S.qready, 0);
    int js = 0, jp = 0;
    uint64_t t_last = globaltimer();
    while (jp < nblk && !*reinterpret_cast<volatile int*>(&S.abort)) {
      bool progress = false;
      if (js < nblk && js <= jp + 1 && mbar_try_wait(&S.kready, js & 1)) {
        tc_fence_after();
        const uint32_t tS = tmem + 128 * (js & 1);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kOpBox + (kk & 3) * 32;
          umma_f16(tS, umma_desc_sw128(qh + off), umma_desc_sw128(kh + off), kCIdesc, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kOpBox + (kk & 3) * 32;
          umma_f16(tS, umma_desc_sw128(qh + off), umma_desc_sw128(kl + off), kCIdesc, true);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kOpBox + (kk & 3) * 32;
          umma_f16(tS, umma_desc_sw128(ql + off), umma_desc_sw128(kh + off), kCIdesc, true);
        }
        umma_commit(&S.sdone[js & 1]);
        ++js;
        progress = true;
      }
      if (jp < js && mbar_try_wait(&S.pready, jp & 1) && mbar_try_wait(&S.vready, jp & 1)) {
        tc_fence_after();
        // A = P from TMEM: K step kk is tokens 16 kk .. 16 kk + 15, columns 8 kk ..
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kOpBox + (kk & 3) * 32;
          umma_f16_ts(tO, tP + 8 * kk, umma_desc_sw128(vh + off), kCIdesc, jp > 0 || kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kOpBox + (kk & 3) * 32;
          umma_f16_ts(tO, tP + 8 * kk, umma_desc_sw128(vl + off), kCIdesc, true);
        }
        umma_commit(&S.pvdone);
        ++jp;
        progress = true;
      }
      if (progress) {
        t_last = globaltimer();
      } else if (globaltimer() - t_last > kCWaitNs) {
        *reinterpret_cast<volatile int*>(&S.abort) = 1;
        report(a.status, KVARN_STATUS_TIMEOUT);
      }
    }
    // every MMA of this thread is complete before TMEM is released
    umma_commit(&S.drain);
    mbar_wait_bounded(&S.drain, 0, kCWaitNs);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kCTmemCols);
}

template <int FMT>
cudaError_t launch_chunk(const ChunkArgs& args, cudaStream_t s) {
  static std::atomic<uint64_t> smem_set{0};
  constexpr int smem = chunk_smem_bytes<FMT>();
  cudaError_t e = ensure_dynamic_smem(chunk_attention_kernel<FMT>, smem, smem_set);
  if (e != cudaSuccess) return e;
  if (args.ntq <= 0 || args.batch <= 0) return cudaSuccess;
  dim3 grid(args.ntq, args.hkv, args.batch);
  chunk_attention_kernel<FMT><<<grid, kCThreads, smem, s>>>(args);
  return cudaGetLastError();
}

}  // namespace

int chunk_rows_per_tile(int g) { return 128 / g; }

cudaError_t launch_chunk_attention(const ChunkArgs& args, cudaStream_t s) {
  if (args.fmt == kFmtM16) return launch_chunk<kFmtM16>(args, s);
  if (args.fmt == kFmtPC) return launch_chunk<kFmtPC>(args, s);
  if (args.fmt == kFmtG64) return launch_chunk<kFmtG64>(args, s);
  if (args.fmt == kFmtV4) return launch_chunk<kFmtV4>(args, s);
  if (args.fmt == kFmtK8) return launch_chunk<kFmtK8>(args, s);
  return launch_chunk<kFmtF32>(args, s);
}

}  // namespace kvarn
