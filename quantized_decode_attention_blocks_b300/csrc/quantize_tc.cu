// quantize_tc.cu -- KVarN-style block quantization of 128-token x 128-channel
// tiles on the fifth-generation tensor cores: Hadamard rotation, Sinkhorn-like
// log-domain variance normalization, asymmetric RTN (K 4-bit, V 2-bit) and
// packing into the page record.
//
// Source of the method: "KVarN: Huawei'den KV-Cache Kuantizasyonu icin Yerel
// vLLM Backend'i" (blog.edumints.com), section "KVarN Nasil Calisir?", stages
// "Dondurulmus Onbellek" (rotation), "Normalize Edilmis Onbellek"
// (normalization) and "Kuantize Edilmis Onbellek" (RTN); format kvarn_k4v2_g128.
//
// Layout of the work.  A persistent CTA runs two independent tile pipelines
// (warpgroups of 128 threads).  For each tile, one thread of the pipeline
// issues the TMA load of the fp16 tile X (two 64-channel boxes, 128-byte
// swizzle) and then two chains of tcgen05.mma against the +-1 Sylvester
// matrix Hs (held once per CTA in shared memory, symmetric):
//     Y  = X Hs      (TMEM lane t = token t, column d = channel d)
//     Y^T = Hs X^T   (TMEM lane d = channel d, column t = token t)
// so that thread t reads its token row and thread d its channel column from
// TMEM without any transpose.  The products of fp16 inputs and +-1 are exact
// and accumulate in fp32; Y = sqrt(128) y with y_t = H x_t, and the factor
// cancels in every normalized quantity (it is removed from the stored s', z').
// The next tile's TMA load runs under this tile's MMAs and arithmetic.
//
// Arithmetic (fp32, centred two-pass moments as in the definition):
//  * row step t:    1/r_t = 1 / std_d(Y_td / c_d)       (the old r_t cancels)
//  * column step d: c_d   = std_t(Y_td / r_t)
//  * a row / column whose variance is <= 1e-10 * its mean square keeps its
//    previous scale;
//  * RTN per token on x_td = Y_td / c_d: s' = (max - min) / (2^b - 1) and
//    z' = min (the row scale r_t cancels from the codes and folds into s', z'),
//    q = rint((x - min) * (2^b - 1) / (max - min)) as one fused multiply-add
//    with 1.5 * 2^23, whose low mantissa bits are then the code.
#include <cuda.h>
#include <stddef.h>

#include "kvarn_internal.cuh"
#include "ptx.cuh"

namespace kvarn {
namespace {

using namespace ptx;

constexpr int kWG = 2;                            // tile pipelines per CTA
constexpr int kWGThreads = 128;                   // one thread per TMEM lane (row)
constexpr int kQThreads = kWGThreads * kWG;
constexpr uint32_t kTileBytes = kT * kD * 2;      // one fp16 tile
constexpr uint32_t kBoxBytes = kTileBytes / 2;    // 64 channels x 128 tokens
constexpr uint32_t kTmemCols = 256 * kWG;         // Y and Y^T per pipeline
constexpr uint64_t kQWaitNs = 2000000000ull;
// instruction descriptor: kind::f16, fp16 A and B (both K-major), fp32 D,
// M = 128, N = 128
constexpr uint32_t kIdesc = (1u << 4) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
constexpr float kMagic = 12582912.0f;             // 1.5 * 2^23
constexpr uint32_t kMagicBits = 0x4B400000u;
// kMagicBits summed over the eight nibble (sixteen crumb) positions of a word
constexpr uint32_t kMagicK = kMagicBits * 0x11111111u;
constexpr uint32_t kMagicV = kMagicBits * 0x55555555u;

// Tile handed from a pipeline's leader thread to its other threads.
struct TileInfo {
  int id;            // tile id, >= ntiles when the pipeline is done
  int part;          // 0: K, 1: V
  long long rec;     // byte offset of the destination record in the pool, -1: none
};

struct __align__(1024) QSmem {
  uint8_t hs[kTileBytes];                // +-1 Sylvester matrix, fp16, swizzled
  uint8_t x[kWG][2][kTileBytes];         // input tiles (then the packed output), 2 stages
  __align__(16) float ra[kWG][kT];       // 1 / r_t, in units of Y
  __align__(16) float cb[kWG][kD];       // 1 / c_d
  __align__(16) float vmin[kWG][kT];     // V: per-token min of x
  __align__(16) float vinv[kWG][kT];     // V: per-token 3 / (max - min)
  __align__(16) float cc[kWG][kD];       // c_d
  TileInfo info[kWG][2];                 // tile held in each stage
  uint64_t xbar[kWG][2];                 // tile landed
  uint64_t mbar[kWG];                    // MMAs done
  uint32_t tmem_base;
};
static_assert(offsetof(QSmem, ra) % 16 == 0 && offsetof(QSmem, cb) % 16 == 0 &&
                  offsetof(QSmem, cc) % 16 == 0 && offsetof(QSmem, vmin) % 16 == 0 &&
                  offsetof(QSmem, vinv) % 16 == 0 && offsetof(QSmem, x) % 1024 == 0 &&
                  offsetof(QSmem, xbar) % 8 == 0,
              "vector loads and barriers need these alignments");

struct QTileArgs {
  int mode;            // 0: the full blocks of a prefill, 1: tails filled by an append
  int batch, hkv, iters, nb, ntiles;
  int roles;           // tensor-map dimension of (head, token, sequence), 2 bits each
  const int32_t* seq_lens;     // mode 0
  const int32_t* pos;          // mode 1: length before the append
  const int32_t* block_table;
  int max_blocks, max_seq;
  uint8_t* pool;
  int64_t num_pages;
  int32_t* status;
};

// One tile of the tile space.  Mode 0: id = ((b * nb + j) * hkv + h) * 2 + part.
// Mode 1: id = (b * hkv + h) * 2 + part; the source is slot 0.. of the tail.
struct Tile {
  int b, j, h, part, t0;
};

__device__ __forceinline__ bool tile_of(const QTileArgs& a, int id, Tile& tl) {
  tl.part = id & 1;
  int rest = id >> 1;
  tl.h = rest % a.hkv;
  rest /= a.hkv;
  if (a.mode == 0) {
    tl.j = rest % a.nb;
    tl.b = rest / a.nb;
    const int len = a.seq_lens[tl.b];
    if (len < 0 || len > a.max_seq) {
      if (tl.j == 0 && tl.h == 0 && tl.part == 0) report(a.status, KVARN_STATUS_BAD_LENGTH);
      return false;
    }
    tl.t0 = kT * tl.j;
    return tl.j < len / kT;
  }
  tl.b = rest;
  const int p = a.pos[tl.b];
  tl.j = p / kT;
  tl.t0 = 0;
  return p >= 0 && p % kT == kT - 1;
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float min3f(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// 64 columns (64 c .. 64 c + 63) of this thread's TMEM lane, scaled in place
// by f (shared memory, the same weights for every thread: broadcast loads)
// when HAS_F.
template <bool HAS_F>
__device__ __forceinline__ void row_chunk(uint32_t taddr, int c, const float* f,
                                          float (&v)[64]) {
  tmem_ld64(taddr + 64 * c, v);
  tmem_wait_ld();
  if (HAS_F) {
#pragma unroll
    for (int i = 0; i < 64; i += 4) {
      const float4 f4 = *reinterpret_cast<const float4*>(f + 64 * c + i);
      const float2 a0 = __fmul2_rn(make_float2(v[i], v[i + 1]), make_float2(f4.x, f4.y));
      const float2 a1 = __fmul2_rn(make_float2(v[i + 2], v[i + 3]), make_float2(f4.z, f4.w));
      v[i] = a0.x;
      v[i + 1] = a0.y;
      v[i + 2] = a1.x;
      v[i + 3] = a1.y;
    }
  }
}

// Centred population moments of w_c = Y[lane][c] f_c over the 128 columns of
// this thread's TMEM lane.  Each half of 64 columns is done in two passes
// over registers with its 64 weights loaded once (the weight loads, shared
// memory broadcasts, are the costly part), and the halves are merged with the
// parallel-variance formula M2 = M2_a + M2_b + (mean_a - mean_b)^2 n_a n_b / n
// (Chan, Golub and LeVeque), which is as stable as one two-pass sweep.  The
// weights are fused into the arithmetic: three FP32 operations per value.
__device__ __forceinline__ void moments_tm(uint32_t taddr, const float* f, float& mean,
                                           float& var) {
  float hm[2], hq[2];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    float v[64], w[64];
    tmem_ld64(taddr + 64 * c, v);
#pragma unroll
    for (int i = 0; i < 64; i += 4) {
      const float4 f4 = *reinterpret_cast<const float4*>(f + 64 * c + i);
      w[i] = f4.x;
      w[i + 1] = f4.y;
      w[i + 2] = f4.z;
      w[i + 3] = f4.w;
    }
    tmem_wait_ld();
    float2 s[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) s[k] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 64; i += 8)
#pragma unroll
      for (int k = 0; k < 4; ++k)
        s[k] = __ffma2_rn(make_float2(v[i + 2 * k], v[i + 2 * k + 1]),
                          make_float2(w[i + 2 * k], w[i + 2 * k + 1]), s[k]);
    const float m = (((s[0].x + s[0].y) + (s[1].x + s[1].y)) +
                     ((s[2].x + s[2].y) + (s[3].x + s[3].y))) * (1.f / 64.f);
    const float2 nm = make_float2(-m, -m);
#pragma unroll
    for (int k = 0; k < 4; ++k) s[k] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 64; i += 8)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float2 e = __ffma2_rn(make_float2(v[i + 2 * k], v[i + 2 * k + 1]),
                                    make_float2(w[i + 2 * k], w[i + 2 * k + 1]), nm);
        s[k] = __ffma2_rn(e, e, s[k]);
      }
    hm[c] = m;
    hq[c] = ((s[0].x + s[0].y) + (s[1].x + s[1].y)) + ((s[2].x + s[2].y) + (s[3].x + s[3].y));
  }
  const float d = hm[0] - hm[1];
  mean = 0.5f * (hm[0] + hm[1]);
  var = (hq[0] + hq[1] + 32.f * d * d) * (1.f / 128.f);
}

// min and max of w_c = Y[lane][c] f_c
__device__ __forceinline__ void minmax_tm(uint32_t taddr, const float* f, float& mn, float& mx) {
  mn = INFINITY;
  mx = -INFINITY;
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    float v[64];
    row_chunk<true>(taddr, c, f, v);
#pragma unroll
    for (int i = 0; i < 64; i += 4) {
      mn = min3f(mn, v[i], v[i + 1]);
      mx = max3f(mx, v[i], v[i + 1]);
      mn = min3f(mn, v[i + 2], v[i + 3]);
      mx = max3f(mx, v[i + 2], v[i + 3]);
    }
  }
}

__device__ __forceinline__ bool keep_scale(float mean, float var) {
  // variance <= 1e-10 * mean square (mean square = var + mean^2): skip
  return !(var > 1e-10f * (var + mean * mean));
}

// +-1 Sylvester matrix element (n, k) as fp16 bits
__device__ __forceinline__ uint32_t hs_bits(int n, int k) {
  return (__popc(n & k) & 1) ? 0xBC00u : 0x3C00u;
}

__global__ void __launch_bounds__(kQThreads, 1)
    quantize_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv, const QTileArgs a) {
  extern __shared__ uint8_t smem_raw[];
  QSmem& S = *reinterpret_cast<QSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, wg = tid / kWGThreads, wt = tid % kWGThreads;
  const int warp = tid >> 5;
  const bool leader = wt == 0;
  const int row = wt;   // this thread's TMEM lane: token in Y, channel in Y^T

  // ---- once per CTA: Hs in the 128-byte swizzled K-major layout (two boxes
  // of 64 columns; 16-byte chunk c of row n sits at chunk c ^ (n & 7)) ----
  for (int i = tid; i < kT * 16; i += kQThreads) {
    const int n = i >> 4, c = i & 15, box = c >> 3, cw = c & 7;
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int k = 8 * c + 2 * e;
      w[e] = hs_bits(n, k) | (hs_bits(n, k + 1) << 16);
    }
    *reinterpret_cast<uint4*>(S.hs + box * kBoxBytes + n * 128 + ((cw ^ (n & 7)) << 4)) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
  fence_proxy_async_smem();
  if (tid == 0) {
#pragma unroll
    for (int g = 0; g < kWG; ++g) {
      mbar_init(&S.xbar[g][0], 1);
      mbar_init(&S.xbar[g][1], 1);
      mbar_init(&S.mbar[g], 1);
    }
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&S.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  const int gw = blockIdx.x * kWG + wg, nw = gridDim.x * kWG;
  const uint32_t dY = tmem + wg * 256, dYT = dY + 128;                  // MMA destinations
  const uint32_t lanes = (uint32_t)(32 * (warp & 3)) << 16;
  const uint32_t tY = dY + lanes, tYT = dYT + lanes;                      // this warp's lanes
  float* const ra = S.ra[wg];
  float* const cb = S.cb[wg];
  float* const cc = S.cc[wg];
  const uint32_t bar_id = 1 + wg;
  const int rh = a.roles & 3, rt = (a.roles >> 2) & 3;   // tensor-map dims of head, token

  // leader only: the next valid tile from `id` on, its TMA load into stage
  // `st`, and its hand-off record for the other threads
  auto prepare = [&](int id, int st) {
    Tile tl;
    while (id < a.ntiles && !tile_of(a, id, tl)) id += nw;
    TileInfo& info = S.info[wg][st];
    info.id = id;
    info.part = 0;
    info.rec = -1;
    if (id >= a.ntiles) return;
    info.part = tl.part;
    const bool in_table = tl.j < a.max_blocks;
    const int64_t page =
        in_table ? (int64_t)a.block_table[(int64_t)tl.b * a.max_blocks + tl.j] : -1;
    if (page >= 0 && page < a.num_pages)
      info.rec = (long long)((page * a.hkv + tl.h) * (int64_t)kRec);
    else
      report(a.status, in_table ? KVARN_STATUS_BAD_PAGE : KVARN_STATUS_BAD_LENGTH);
    const CUtensorMap* tm = tl.part ? &tmv : &tmk;
    const int c1 = rh == 1 ? tl.h : rt == 1 ? tl.t0 : tl.b;
    const int c2 = rh == 2 ? tl.h : rt == 2 ? tl.t0 : tl.b;
    const int c3 = rh == 3 ? tl.h : rt == 3 ? tl.t0 : tl.b;
    bulk_wait_read();   // an earlier tile's packed output may still be leaving this stage
    uint64_t* bar = &S.xbar[wg][st];
    mbar_arrive_expect_tx(bar, kTileBytes);
    tma_load_4d(S.x[wg][st], tm, 0, c1, c2, c3, bar);
    tma_load_4d(S.x[wg][st] + kBoxBytes, tm, 64, c1, c2, c3, bar);
  };

  if (leader) prepare(gw, 0);
  named_sync(bar_id, kWGThreads);
  int stage = 0;
  uint32_t xph0 = 0, xph1 = 0, mph = 0;

  while (true) {
    const TileInfo cur = S.info[wg][stage];
    if (cur.id >= a.ntiles) break;
    uint8_t* const xs = S.x[wg][stage];
    {
      const uint32_t ph = stage ? xph1 : xph0;
      if (!mbar_wait_bounded(&S.xbar[wg][stage], ph, kQWaitNs) && leader)
        report(a.status, KVARN_STATUS_TIMEOUT);
    }
    if (stage) xph1 ^= 1; else xph0 ^= 1;
    if (leader) {
      tc_fence_after();
      const uint32_t xa = smem_u32(xs), ha = smem_u32(S.hs);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {   // Y = X Hs: A = X (tokens x channels), B = Hs
        const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
        umma_f16(dY, umma_desc_sw128(xa + off), umma_desc_sw128(ha + off), kIdesc, kk > 0);
      }
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {   // Y^T = Hs X^T: A = Hs, B = X
        const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
        umma_f16(dYT, umma_desc_sw128(ha + off), umma_desc_sw128(xa + off), kIdesc, kk > 0);
      }
      umma_commit(&S.mbar[wg]);
      // the next tile of this pipeline, loading while this one is processed
      prepare(cur.id + nw, stage ^ 1);
    }
    const int part = cur.part;

    // ---- first row step from X itself, while the MMAs run: the rotated row
    // y = Hs x / sqrt(128) has mean x_0 / sqrt(128) and variance
    // sum_{k >= 1} x_k^2 / 128 (Hs has orthogonal rows of norm^2 128, and
    // column sums 128, 0, 0, ...); in units of Y = Hs x: mean x_0, variance
    // sum_{k >= 1} x_k^2 ----
    cb[row] = 1.f;
    cc[row] = 1.f;
    if (a.iters > 0) {
      float2 s2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                      make_float2(0.f, 0.f)};
      float x0 = 0.f;
#pragma unroll
      for (int c = 0; c < 16; ++c) {   // 16-byte chunk c: channels 8c .. 8c + 7
        const uint8_t* xr = xs + (c >> 3) * kBoxBytes + row * 128;
        uint4 u = *reinterpret_cast<const uint4*>(xr + (((c & 7) ^ (row & 7)) << 4));
        if (c == 0) {
          x0 = __half2float(__ushort_as_half((unsigned short)(u.x & 0xFFFFu)));
          u.x &= 0xFFFF0000u;   // channel 0 is the mean, not part of the variance
        }
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
          s2[e] = __ffma2_rn(f, f, s2[e]);
        }
      }
      const float var = ((s2[0].x + s2[0].y) + (s2[1].x + s2[1].y)) +
                        ((s2[2].x + s2[2].y) + (s2[3].x + s2[3].y));
      ra[row] = keep_scale(x0, var) ? kInvSqrt128 : rsqrtf(var);
    } else {
      ra[row] = kInvSqrt128;
    }
    named_sync(bar_id, kWGThreads);
    if (!mbar_wait_bounded(&S.mbar[wg], mph, kQWaitNs) && leader)
      report(a.status, KVARN_STATUS_TIMEOUT);
    mph ^= 1;
    tc_fence_after();

    // ---- Sinkhorn-like normalization: column step (row = channel), then
    // for the later iterations row step (row = token) and column step ----
    for (int it = 0; it < a.iters; ++it) {
      if (it > 0) {
        float mean, var;
        moments_tm(tY, cb, mean, var);
        if (!keep_scale(mean, var)) ra[row] = rsqrtf(var);
        named_sync(bar_id, kWGThreads);
      }
      float mean, var;
      moments_tm(tYT, ra, mean, var);
      if (!keep_scale(mean, var)) {
        const float rs = rsqrtf(var);
        cc[row] = var * rs;
        cb[row] = rs;
      }
      named_sync(bar_id, kWGThreads);
    }

    // ---- RTN + pack into the staging copy of the record part (the smem of
    // this tile's input, free now), written out by one bulk copy ----
    uint8_t* const out = xs;
    const float2 mg = make_float2(kMagic, kMagic);
    if (part == 0) {
      // K: token-major, 64 bytes per token; nibble e of word w = channel 8w + e
      float mn, mx;
      minmax_tm(tY, cb, mn, mx);
      const float range = mx - mn;
      const float inv = range > 0.f ? __fdividef(15.f, range) : 0.f;
      *reinterpret_cast<float2*>(out + kOffKSZ + 8 * row) =
          make_float2(range * (kInvSqrt128 / 15.f), mn * kInvSqrt128);
      reinterpret_cast<float*>(out + kOffKC)[row] = cc[row];
      // u = (y c^-1 - min) (15 / range): y c^-1 - min in one rounding
      const float2 nm = make_float2(-mn, -mn), iv = make_float2(inv, inv);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float v[64];
        row_chunk<false>(tY, c, nullptr, v);
        uint32_t w[8];
#pragma unroll
        for (int wd = 0; wd < 8; ++wd) {
          uint32_t acc = 0u - kMagicK;
          const float4 c0 = *reinterpret_cast<const float4*>(cb + 64 * c + 8 * wd);
          const float4 c1 = *reinterpret_cast<const float4*>(cb + 64 * c + 8 * wd + 4);
          const float cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const int d = 8 * wd + e;
            const float2 dd = __ffma2_rn(make_float2(v[d], v[d + 1]),
                                         make_float2(cw[e], cw[e + 1]), nm);
            const float2 f = __ffma2_rn(dd, iv, mg);
            acc += __float_as_uint(f.x) << (4 * e);
            acc += __float_as_uint(f.y) << (4 * e + 4);
          }
          w[wd] = acc;
        }
        // rows of 64 bytes: start at a chunk that depends on the row so that
        // eight consecutive threads hit different banks
        uint4* dst = reinterpret_cast<uint4*>(out + kOffKCodes + 64 * row + 32 * c);
        const int sw = row & 1;
        dst[sw] = make_uint4(w[4 * sw], w[4 * sw + 1], w[4 * sw + 2], w[4 * sw + 3]);
        dst[sw ^ 1] = make_uint4(w[4 * (sw ^ 1)], w[4 * (sw ^ 1) + 1], w[4 * (sw ^ 1) + 2],
                                 w[4 * (sw ^ 1) + 3]);
      }
    } else {
      // V: publish the per-token min and 3 / range, then thread d packs channel d
      float mn, mx;
      minmax_tm(tY, cb, mn, mx);
      const float range = mx - mn;
      const float inv = range > 0.f ? __fdividef(3.f, range) : 0.f;
      S.vmin[wg][row] = mn;
      S.vinv[wg][row] = inv;
      *reinterpret_cast<float2*>(out + (kOffVSZ - kKPart) + 8 * row) =
          make_float2(range * (kInvSqrt128 / 3.f), mn * kInvSqrt128);
      reinterpret_cast<float*>(out + (kOffVC - kKPart))[row] = cc[row];
      named_sync(bar_id, kWGThreads);
      const float cd = cb[row];
      const float2 cd2 = make_float2(cd, cd);
      const float* vm = S.vmin[wg];
      const float* vi = S.vinv[wg];
      uint32_t acc[4][2];
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[j][0] = acc[j][1] = 0u - kMagicV;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float v[64];
        row_chunk<false>(tYT, c, nullptr, v);
#pragma unroll
        for (int i = 0; i < 64; i += 4) {
          const int tt = 64 * c + i;
          const float4 m4 = *reinterpret_cast<const float4*>(vm + tt);
          const float4 i4 = *reinterpret_cast<const float4*>(vi + tt);
          const float2 d0 = __ffma2_rn(make_float2(v[i], v[i + 1]), cd2,
                                       make_float2(-m4.x, -m4.y));
          const float2 d1 = __ffma2_rn(make_float2(v[i + 2], v[i + 3]), cd2,
                                       make_float2(-m4.z, -m4.w));
          const float2 f0 = __ffma2_rn(d0, make_float2(i4.x, i4.y), mg);
          const float2 f1 = __ffma2_rn(d1, make_float2(i4.z, i4.w), mg);
          const float fv[4] = {f0.x, f0.y, f1.x, f1.y};
#pragma unroll
          for (int s2 = 0; s2 < 4; ++s2) {
            const int tok = tt + s2;
            const int k = tok >> 4, fh = (tok >> 3) & 1, j = (tok >> 1) & 3, sb = tok & 1;
            const int crumb = 2 * (k & 3) + fh + 8 * sb;
            acc[j][k >> 2] += __float_as_uint(fv[s2]) << (2 * crumb);
          }
        }
      }
      uint32_t* vw = reinterpret_cast<uint32_t*>(out + (kOffVCodes - kKPart));
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint2*>(vw + v_word(row, j, 0)) = make_uint2(acc[j][0], acc[j][1]);
    }
    // the staging copy is complete and TMEM is free for the next tile
    fence_proxy_async_smem();
    tc_fence_before();
    named_sync(bar_id, kWGThreads);
    if (leader && cur.rec >= 0) {
      bulk_s2g(a.pool + cur.rec + (part ? kKPart : 0), out, part ? kVPart : kKPart);
      bulk_commit();
    }
    stage ^= 1;
  }

  // ---- teardown: every MMA was waited for; the packed outputs are written
  // before the CTA's shared memory is released; free TMEM ----
  if (leader) bulk_wait_all();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// Leftover tokens (len mod 128) of every sequence copied to its tail buffer.
// grid: (2 * hkv, batch); block 128.
__global__ void __launch_bounds__(128) tail_copy_kernel(QuantizeArgs a) {
  const int b = blockIdx.y, h = blockIdx.x >> 1, part = blockIdx.x & 1;
  const int len = a.seq_lens[b];
  if (len < 0 || len > a.max_seq) return;
  const int nfull = len / kT, rem = len % kT;
  const __half* src = (part ? a.v : a.k) + (int64_t)b * a.sb + (int64_t)h * a.sh;
  __half* tail = (part ? a.tail_v : a.tail_k) + ((int64_t)b * a.hkv + h) * kT * kD;
  for (int i = threadIdx.x; i < rem * (kD / 8); i += blockDim.x) {
    const int r = i / (kD / 8), c = i % (kD / 8);
    const uint4* s4 = reinterpret_cast<const uint4*>(src + ((int64_t)nfull * kT + r) * a.st);
    reinterpret_cast<uint4*>(tail + (int64_t)r * kD)[c] = __ldg(s4 + c);
  }
}

// Decode-time append: token pos[b] into tail slot pos % 128.  grid: (2 * hkv,
// batch); block 32 (16 lanes copy the 256 bytes).
__global__ void __launch_bounds__(32) append_copy_kernel(AppendArgs a) {
  const int b = blockIdx.y, h = blockIdx.x >> 1, part = blockIdx.x & 1;
  const int p = a.pos[b];
  if (p < 0) return;
  const int slot = p % kT;
  __half* tail = (part ? a.tail_v : a.tail_k) + ((int64_t)b * a.hkv + h) * kT * kD;
  const __half* src = (part ? a.v_new : a.k_new) + ((int64_t)b * a.hkv + h) * kD;
  if (threadIdx.x < kD / 8)
    reinterpret_cast<uint4*>(tail + (int64_t)slot * kD)[threadIdx.x] =
        __ldg(reinterpret_cast<const uint4*>(src) + threadIdx.x);
}

// ------------------------------------------------------------- host side --

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Tensor map over an fp16 tensor whose element (b, t, h, c) sits at
// b*sb + t*st + h*sh + c (elements), boxes of 64 channels x 128 tokens of one
// (head, sequence).  The three outer dimensions are ordered by stride; *roles
// receives which map dimension holds the head (bits 0-1) and the token (2-3).
bool encode_tile_map(CUtensorMap* map, const void* base, int64_t sb, int64_t st, int64_t sh,
                     int batch, int tokens, int hkv, int* roles) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  struct Dim {
    int64_t stride, extent;
    int role;   // 0 head, 1 token, 2 sequence
  } d[3] = {{sh, hkv, 0}, {st, tokens, 1}, {sb, batch, 2}};
  for (int i = 0; i < 3; ++i)
    for (int k = i + 1; k < 3; ++k)
      if (d[k].stride < d[i].stride) {
        Dim tmp = d[i];
        d[i] = d[k];
        d[k] = tmp;
      }
  cuuint64_t dims[4] = {(cuuint64_t)kD, 0, 0, 0};
  cuuint64_t strides[3];
  cuuint32_t box[4] = {64, 1, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  int r = 0;
  for (int i = 0; i < 3; ++i) {
    dims[i + 1] = (cuuint64_t)(d[i].extent > 0 ? d[i].extent : 1);
    strides[i] = (cuuint64_t)(d[i].stride > 0 ? d[i].stride : kD) * 2;
    if (d[i].role == 1) box[i + 1] = kT;
    if (d[i].role == 0) r |= (i + 1);
    if (d[i].role == 1) r |= (i + 1) << 2;
  }
  *roles = r;
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

constexpr int kQSmemBytes = (int)sizeof(QSmem) + 1024;

cudaError_t launch_tiles(const CUtensorMap& mk, const CUtensorMap& mv, const QTileArgs& qa,
                         cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(quantize_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  if (qa.ntiles <= 0) return cudaSuccess;
  const int want = (qa.ntiles + kWG - 1) / kWG;
  const int grid = want < kNumSMs ? want : kNumSMs;
  quantize_tc_kernel<<<grid, kQThreads, kQSmemBytes, s>>>(mk, mv, qa);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize_blocks(const QuantizeArgs& a, cudaStream_t s) {
  QTileArgs qa{};
  qa.mode = 0;
  qa.batch = a.batch;
  qa.hkv = a.hkv;
  qa.iters = a.iters;
  qa.nb = a.max_seq / kT;
  qa.ntiles = a.batch * qa.nb * a.hkv * 2;
  qa.seq_lens = a.seq_lens;
  qa.block_table = a.block_table;
  qa.max_blocks = a.max_blocks;
  qa.max_seq = a.max_seq;
  qa.pool = a.pool;
  qa.num_pages = a.num_pages;
  qa.status = a.status;
  if (qa.ntiles > 0) {
    CUtensorMap mk, mv;
    int rk = 0, rv = 0;
    if (!encode_tile_map(&mk, a.k, a.sb, a.st, a.sh, a.batch, a.max_seq, a.hkv, &rk) ||
        !encode_tile_map(&mv, a.v, a.sb, a.st, a.sh, a.batch, a.max_seq, a.hkv, &rv) || rk != rv)
      return cudaErrorInvalidValue;
    qa.roles = rk;
    cudaError_t e = launch_tiles(mk, mv, qa, s);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(2 * a.hkv, a.batch);
  tail_copy_kernel<<<grid, 128, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_append_token(const AppendArgs& a, cudaStream_t s) {
  dim3 grid(2 * a.hkv, a.batch);
  append_copy_kernel<<<grid, 32, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // tails whose block just filled: same kernel as the prefill, reading the tail
  // buffers [B][Hkv][128][128]
  QTileArgs qa{};
  qa.mode = 1;
  qa.batch = a.batch;
  qa.hkv = a.hkv;
  qa.iters = a.iters;
  qa.nb = 1;
  qa.ntiles = a.batch * a.hkv * 2;
  qa.pos = a.pos;
  qa.block_table = a.block_table;
  qa.max_blocks = a.max_blocks;
  qa.max_seq = 0;
  qa.pool = a.pool;
  qa.num_pages = a.num_pages;
  qa.status = a.status;
  CUtensorMap mk, mv;
  int rk = 0, rv = 0;
  const int64_t sh = (int64_t)kT * kD, sb = sh * a.hkv;
  if (!encode_tile_map(&mk, a.tail_k, sb, kD, sh, a.batch, kT, a.hkv, &rk) ||
      !encode_tile_map(&mv, a.tail_v, sb, kD, sh, a.batch, kT, a.hkv, &rv))
    return cudaErrorInvalidValue;
  qa.roles = rk;
  return launch_tiles(mk, mv, qa, s);
}

}  // namespace kvarn
