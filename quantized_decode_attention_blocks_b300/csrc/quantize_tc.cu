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
// of 256 threads.  For each tile, one thread of the pipeline has issued the
// TMA load of the fp16 tile X (two 64-channel boxes, 128-byte swizzle) a tile
// ahead; another issues two chains of tcgen05.mma against the +-1 Sylvester
// matrix Hs (held once per CTA in shared memory, symmetric, its rows in the
// order chan_of):
//     Y  = X Hs      (TMEM lane t = token t, column n = channel chan_of(n))
//     Y^T = Hs X^T   (TMEM lane n = channel chan_of(n), column t = token t)
// The products of fp16 inputs and +-1 are exact and accumulate in fp32;
// Y = sqrt(128) y with y_t = H x_t, and the factor cancels in every normalized
// quantity (it is removed from the stored s', z').
//
// Each warp reads 16 TMEM lanes of Y or Y^T in the 16x256b shape: a thread
// holds two rows, 32 columns of each, and the four threads of a quad hold one
// row's 128 columns.  Row statistics are quad reductions, and each thread
// needs only the 32 weights of its columns (the other axis's scales), so the
// shared-memory traffic of the weights is a quarter of a thread-per-row
// layout's.  The column order chan_of makes a thread's 32 columns of Y the
// consecutive channels of whole K code words, and its 32 columns of Y^T
// (tokens) whole V code words, so that every thread packs complete words.
//
// Arithmetic (fp32, centred two-pass moments as in the definition):
//  * row step t:    1/r_t = 1 / std_d(Y_td / c_d)       (the old r_t cancels)
//  * column step d: c_d   = std_t(Y_td / r_t)
//  * a row / column whose variance is <= 1e-10 * its mean square keeps its
//    previous scale;
//  * the "_rms" variant divides by the root mean square (mean^2 + variance)
//    instead of the std, and keeps the scale only of an all-zero row / column;
//  * RTN per token on x_td = Y_td / c_d: s' = (max - min) / (2^b - 1) and
//    z' = min (the row scale r_t cancels from the codes and folds into s', z'),
//    q = rint((x - min) * (2^b - 1) / (max - min)) as one fused multiply-add
//    with 1.5 * 2^23, whose low mantissa bits are then the code.
#include <cuda.h>
#include <stddef.h>
#include <string.h>

#include "kvarn_internal.cuh"
#include "ptx.cuh"

namespace kvarn {
namespace {

using namespace ptx;

constexpr int kWG = 2;                            // tile pipelines per CTA
// 256 threads per pipeline: warp w of a pipeline reads the TMEM lane quarter
// w & 3, and the 16-lane half w >> 2 of it
constexpr int kWGThreads = 256;
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
// kMagicBits summed over the eight nibble (sixteen crumb, four byte)
// positions of a word
constexpr uint32_t kMagicK = kMagicBits * 0x11111111u;
constexpr uint32_t kMagicB = kMagicBits * 0x01010101u;
constexpr uint32_t kMagicV = kMagicBits * 0x55555555u;

// Tile handed from a pipeline's leader thread to its other threads.
struct TileInfo {
  int id;            // tile id, >= ntiles when the pipeline is done
  int part;          // 0: K, 1: V
  long long rec;     // byte offset of the destination record in the pool, -1: none
};

struct __align__(1024) QSmem {
  uint8_t hs[kTileBytes];                // +-1 Sylvester matrix, fp16, swizzled
  uint8_t x[kWG][2][kTileBytes];         // input tiles, 2 stages per pipeline
  __align__(128) uint8_t out[kWG][RecFmt<kFmtK8>::kpart];   // packed record part (the
                                                            // largest), staged for the bulk store
  __align__(16) float ra[kWG][kT];       // 1 / r_t, in units of Y
  float r1part[kWG][2][kT];              // first row step of the next tile: half sums
  float r1x0[kWG][kT];                   //   and channel 0
  __align__(16) float cb[kWG][kD];       // 1 / c, indexed by Y column (channel chan_of(n))
  __align__(16) float vmin[kWG][2 * kT]; // V: per-token (and group) min of x
  __align__(16) float vinv[kWG][2 * kT]; // V: per-token (and group) 3 / (max - min)
  __align__(16) float cc[kWG][kD];       // c_d, natural channel order
  TileInfo info[kWG][2];                 // tile held in each stage
  uint64_t full[kWG][2];                 // stage loaded (producer -> pipeline)
  uint64_t mbar[kWG];                    // MMAs done
  uint32_t tmem_base;
  int abort;                             // a bounded wait ran out: stop waiting
};
static_assert(offsetof(QSmem, ra) % 16 == 0 && offsetof(QSmem, cb) % 16 == 0 &&
                  offsetof(QSmem, cc) % 16 == 0 && offsetof(QSmem, vmin) % 16 == 0 &&
                  offsetof(QSmem, vinv) % 16 == 0 && offsetof(QSmem, x) % 1024 == 0 &&
                  offsetof(QSmem, out) % 128 == 0 && offsetof(QSmem, full) % 8 == 0,
              "vector loads, bulk copies and barriers need these alignments");

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
  int rms;             // Sinkhorn statistic: 0 centred std, 1 uncentred RMS ("_rms")
};

// The plain copies folded into the same launch: mode 0 copies every
// sequence's leftover len % 128 tokens to its tail, mode 1 copies the new
// token into tail slot pos % 128.
struct QCopyArgs {
  const __half* src_k;         // mode 0: k, v with strides sb, st, sh; mode 1: k_new, v_new
  const __half* src_v;
  int64_t sb, st, sh;
  __half* tail_k;
  __half* tail_v;
};

// One tile of the tile space.  Mode 0: id = ((b * nb + j) * hkv + h) * 2 + part.
// Mode 1: id = (b * hkv + h) * 2 + part; the source is slot 0.. of the tail.
struct Tile {
  int b, j, h, part, t0;
};

// (b, j, h, part) of tile id from the id alone
__device__ __forceinline__ void tile_decode(const QTileArgs& a, int id, Tile& tl) {
  tl.part = id & 1;
  int rest = id >> 1;
  tl.h = rest % a.hkv;
  rest /= a.hkv;
  if (a.mode == 0) {
    tl.j = rest % a.nb;
    tl.b = rest / a.nb;
  } else {
    tl.b = rest;
  }
}

// Whether the decoded tile is a block to quantize, given its sequence's length
// (mode 0) or length before the append (mode 1).
__device__ __forceinline__ bool tile_valid(const QTileArgs& a, Tile& tl, int len) {
  if (a.mode == 0) {
    if (len < 0 || len > a.max_seq) {
      if (tl.j == 0 && tl.h == 0 && tl.part == 0) report(a.status, KVARN_STATUS_BAD_LENGTH);
      return false;
    }
    tl.t0 = kT * tl.j;
    return tl.j < len / kT;
  }
  tl.j = len / kT;
  tl.t0 = 0;
  return len >= 0 && len % kT == kT - 1;
}

// Metadata of a candidate tile, loaded one tile ahead of its use: the length
// of its sequence and (mode 0) its block-table entry.
struct Cand {
  int id, len, page;
};

__device__ __forceinline__ Cand fetch_cand(const QTileArgs& a, int id) {
  Cand c{id, -1, -1};
  if (id >= a.ntiles) return c;
  Tile tl;
  tile_decode(a, id, tl);
  if (a.mode == 0) {
    c.len = __ldg(a.seq_lens + tl.b);
    if (tl.j < a.max_blocks) c.page = __ldg(a.block_table + (int64_t)tl.b * a.max_blocks + tl.j);
  } else {
    c.len = __ldg(a.pos + tl.b);
  }
  return c;
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

// Channel held by column n of Y and by lane n of Y^T.  The rows of the Hadamard
// operand are stored in this order, so that the columns 8k + 2 (i & 3) + b of
// the 16x256b fragment of thread i are the 32 consecutive channels
// 32 (i & 3) + 2k + b: whole bytes and words of a packed K row.
__device__ __forceinline__ int chan_of(int n) {
  return 32 * ((n >> 1) & 3) + 2 * (n >> 3) + (n & 1);
}

// sums, minima and maxima over the four threads of a quad (one fragment row)
__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  return x + __shfl_xor_sync(0xffffffffu, x, 2);
}
__device__ __forceinline__ float quad_min(float x) {
  x = fminf(x, __shfl_xor_sync(0xffffffffu, x, 1));
  return fminf(x, __shfl_xor_sync(0xffffffffu, x, 2));
}
__device__ __forceinline__ float quad_max(float x) {
  x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 1));
  return fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 2));
}

// Minimum and maximum over the threads holding one RTN group of a fragment
// row: the quad (128 channels), or a pair of it (groups of 64 channels).
template <bool G64>
__device__ __forceinline__ float grp_min(float x) {
  if constexpr (G64) return fminf(x, __shfl_xor_sync(0xffffffffu, x, 1));
  else return quad_min(x);
}
template <bool G64>
__device__ __forceinline__ float grp_max(float x) {
  if constexpr (G64) return fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 1));
  else return quad_max(x);
}

// The weights of this thread's fragment columns 8k + 2q + b (f indexed by
// column): 32 of the 128, one 8-byte load per k.
__device__ __forceinline__ void frag_weights(const float* f, int q, float2 (&w)[16]) {
#pragma unroll
  for (int k = 0; k < 16; ++k) w[k] = *reinterpret_cast<const float2*>(f + 8 * k + 2 * q);
}

__device__ __forceinline__ float2 pair(const float (&v)[64], int k, int e) {
  return make_float2(v[4 * k + 2 * e], v[4 * k + 2 * e + 1]);
}

// Centred population moments, over the 128 columns, of v * w in the two rows
// (e = 0, 1) of this thread's fragment: two passes over registers, the four
// threads of a quad adding their partial sums after each.
__device__ __forceinline__ void frag_moments(const float (&v)[64], const float2 (&w)[16],
                                             float (&mean)[2], float (&var)[2]) {
  float2 s[2][2];
#pragma unroll
  for (int e = 0; e < 2; ++e) s[e][0] = s[e][1] = make_float2(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < 16; ++k)
#pragma unroll
    for (int e = 0; e < 2; ++e) s[e][k & 1] = __ffma2_rn(pair(v, k, e), w[k], s[e][k & 1]);
  float2 nm[2];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    mean[e] = quad_sum((s[e][0].x + s[e][0].y) + (s[e][1].x + s[e][1].y)) * (1.f / 128.f);
    nm[e] = make_float2(-mean[e], -mean[e]);
    s[e][0] = s[e][1] = make_float2(0.f, 0.f);
  }
#pragma unroll
  for (int k = 0; k < 16; ++k)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float2 d = __ffma2_rn(pair(v, k, e), w[k], nm[e]);
      s[e][k & 1] = __ffma2_rn(d, d, s[e][k & 1]);
    }
#pragma unroll
  for (int e = 0; e < 2; ++e)
    var[e] = quad_sum((s[e][0].x + s[e][0].y) + (s[e][1].x + s[e][1].y)) * (1.f / 128.f);
}

__device__ __forceinline__ int lane4(int tid) { return tid & 3; }

// Mode 1: copies the new token of every candidate tile of this CTA (pipeline
// tiles blockIdx.x * kWG + wg + k * nw, i.e. (sequence, head, part)) into its
// tail slot pos % 128; 16 threads per 256-byte row.  Returns whether one of
// them filled its block (slot 127), i.e. whether the CTA has a tile to
// quantize.  The writes are made visible to the TMA engine (async proxy)
// before the CTA's barrier that follows.
__device__ __forceinline__ bool append_copy(const QTileArgs& a, const QCopyArgs& cp, int nw) {
  int fills = 0;
  for (int i = threadIdx.x;; i += blockDim.x) {
    const int ci = i >> 4, c = i & 15;
    const int id = blockIdx.x * kWG + (ci & 1) + (ci >> 1) * nw;   // increasing in ci
    if (id >= a.ntiles) break;
    const int part = id & 1, bh = id >> 1;                      // bh = b * hkv + h
    const int p = __ldg(a.pos + bh / a.hkv);
    if (p < 0) continue;
    const __half* src = (part ? cp.src_v : cp.src_k) + (int64_t)bh * kD;
    __half* dst = (part ? cp.tail_v : cp.tail_k) + ((int64_t)bh * kT + p % kT) * kD;
    reinterpret_cast<uint4*>(dst)[c] = __ldg(reinterpret_cast<const uint4*>(src) + c);
    if (c == 0 && p % kT == kT - 1) fills = 1;
  }
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return fills != 0;
}

// Mode 0: the leftover len % 128 tokens of every (sequence, head, part) to the
// tail buffer, 16-byte chunks spread over the whole grid (grid-stride).
__device__ __forceinline__ void tail_copy(const QTileArgs& a, const QCopyArgs& cp) {
  const int64_t rows = (int64_t)a.batch * a.hkv * 2 * kT;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < rows * 16;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(i & 15);
    const int64_t row = i >> 4;
    const int r = (int)(row % kT);
    const int64_t unit = row / kT;                  // (b * hkv + h) * 2 + part
    const int part = (int)(unit & 1);
    const int64_t bh = unit >> 1;
    const int b = (int)(bh / a.hkv), h = (int)(bh % a.hkv);
    const int len = __ldg(a.seq_lens + b);
    if (len < 0 || len > a.max_seq || r >= len % kT) continue;
    const __half* src = (part ? cp.src_v : cp.src_k) + (int64_t)b * cp.sb + (int64_t)h * cp.sh +
                        ((int64_t)(len / kT) * kT + r) * cp.st;
    __half* dst = (part ? cp.tail_v : cp.tail_k) + (bh * kT + r) * kD;
    reinterpret_cast<uint4*>(dst)[c] = __ldg(reinterpret_cast<const uint4*>(src) + c);
  }
}

__device__ __forceinline__ bool keep_scale(float mean, float var) {
  // variance <= 1e-10 * mean square (mean square = var + mean^2): skip
  return !(var > 1e-10f * (var + mean * mean));
}

// The statistic a step divides by, as its square: the centred variance, or
// for the "_rms" variant the mean square (= variance + mean^2), and whether
// the step applies (centred: not for a (near-)constant row or column; RMS:
// not for an all-zero one).
__device__ __forceinline__ bool step_stat(bool rms, float mean, float var, float& sq) {
  if (rms) {
    sq = fmaf(mean, mean, var);
    return sq > 0.f;
  }
  sq = var;
  return !keep_scale(mean, var);
}

// +-1 Sylvester matrix element (n, k) as fp16 bits
__device__ __forceinline__ uint32_t hs_bits(int n, int k) {
  return (__popc(n & k) & 1) ? 0xBC00u : 0x3C00u;
}

// FMT: the record format (RecFmt): fp32 or fp16 ("_m16") metadata with
// per-token groups, or per-channel groups ("_pc").
template <int FMT>
__global__ void __launch_bounds__(kQThreads, 1)
    quantize_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv, const QTileArgs a,
                       const __grid_constant__ QCopyArgs cp) {
  extern __shared__ uint8_t smem_raw[];
  QSmem& S = *reinterpret_cast<QSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, wg = tid / kWGThreads, wt = tid % kWGThreads;
  const int warp = tid >> 5;
  const int nw = gridDim.x * kWG;
  // the plain copies of this launch; a CTA with no block to quantize leaves
  // before it sets anything up
  if (a.mode == 1) {
    if (!__syncthreads_or(append_copy(a, cp, nw))) return;
  } else if (a.ntiles == 0) {
    tail_copy(a, cp);
    return;
  }
  // roles in a pipeline: wt 0 issues the bulk stores of the packed output;
  // lane 0 of warps 4 and 5 (idle during the first row step, which warps 0-3
  // do) issue the tile's MMAs and the next tile's load
  const bool leader = wt == 0;
  const bool mma_thread = wt == 128;
  const bool load_thread = wt == 160;
  const int row = wt & 127;   // first row step, copies: token or channel
  const bool lower = wt < 128;

  // ---- once per CTA: Hs with its rows in chan_of order, in the 128-byte
  // swizzled K-major layout (two boxes of 64 columns; 16-byte chunk c of row n
  // sits at chunk c ^ (n & 7)) ----
  for (int i = tid; i < kT * 16; i += kQThreads) {
    const int n = i >> 4, c = i & 15, box = c >> 3, cw = c & 7;
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int k = 8 * c + 2 * e;
      w[e] = hs_bits(chan_of(n), k) | (hs_bits(chan_of(n), k + 1) << 16);
    }
    *reinterpret_cast<uint4*>(S.hs + box * kBoxBytes + n * 128 + ((cw ^ (n & 7)) << 4)) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
  fence_proxy_async_smem();
  if (tid == 0) {
#pragma unroll
    for (int g = 0; g < kWG; ++g) {
      mbar_init(&S.full[g][0], 1);
      mbar_init(&S.full[g][1], 1);
      mbar_init(&S.mbar[g], 1);
    }
    S.abort = 0;
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

  const int rh = a.roles & 3, rt = (a.roles >> 2) & 3;   // tensor-map dims of head, token
  // bounded waits; once one has run out every later wait is skipped, so that
  // the kernel still ends (with KVARN_STATUS_TIMEOUT reported)
  auto wait = [&](uint64_t* bar, uint32_t ph) {
    if (*reinterpret_cast<volatile int*>(&S.abort)) return;
    if (!mbar_wait_bounded(bar, ph, kQWaitNs)) {
      *reinterpret_cast<volatile int*>(&S.abort) = 1;
      report(a.status, KVARN_STATUS_TIMEOUT);
    }
  };

  // load thread only: the next valid tile from the candidate on, its TMA load into
  // stage `st` (free: its last tile's MMAs and first row step are done), and
  // its hand-off record for the other threads.  The candidate's metadata was
  // loaded a tile earlier; a candidate that is not a block falls back to a
  // walk with fresh loads.  Returns the id taken (>= ntiles: none).
  auto prepare = [&](Cand c, int st) -> int {
    int id = c.id;
    Tile tl;
    int len = c.len;
    int64_t page = c.page;
    bool ok = false;
    if (id < a.ntiles) {
      tile_decode(a, id, tl);
      ok = tile_valid(a, tl, len);
    }
    if (!ok && id < a.ntiles) {
      for (id += nw; id < a.ntiles; id += nw) {
        const Cand f = fetch_cand(a, id);
        tile_decode(a, id, tl);
        if (tile_valid(a, tl, f.len)) {
          page = f.page;
          ok = true;
          break;
        }
      }
    }
    TileInfo& info = S.info[wg][st];
    info.id = id;
    info.part = 0;
    info.rec = -1;
    if (id >= a.ntiles) return id;
    info.part = tl.part;
    const bool in_table = tl.j < a.max_blocks;
    if (a.mode != 0)
      page = in_table ? (int64_t)a.block_table[(int64_t)tl.b * a.max_blocks + tl.j] : -1;
    if (in_table && page >= 0 && page < a.num_pages)
      info.rec = (long long)((page * a.hkv + tl.h) * (int64_t)RecFmt<FMT>::bytes);
    else
      report(a.status, in_table ? KVARN_STATUS_BAD_PAGE : KVARN_STATUS_BAD_LENGTH);
    const CUtensorMap* tm = tl.part ? &tmv : &tmk;
    const int c1 = rh == 1 ? tl.h : rt == 1 ? tl.t0 : tl.b;
    const int c2 = rh == 2 ? tl.h : rt == 2 ? tl.t0 : tl.b;
    const int c3 = rh == 3 ? tl.h : rt == 3 ? tl.t0 : tl.b;
    uint64_t* bar = &S.full[wg][st];
    mbar_arrive_expect_tx(bar, kTileBytes);
    tma_load_4d(S.x[wg][st], tm, 0, c1, c2, c3, bar);
    tma_load_4d(S.x[wg][st] + kBoxBytes, tm, 64, c1, c2, c3, bar);
    return id;
  };

  const uint32_t dY = tmem + wg * 256, dYT = dY + 128;                  // MMA destinations
  // this warp's 16 TMEM lanes: quarter warp & 3, half (warp >> 2) & 1
  const int hl = (warp >> 2) & 1;
  const uint32_t lanes = (uint32_t)(32 * (warp & 3) + 16 * hl) << 16;
  const uint32_t tY = dY + lanes, tYT = dYT + lanes;
  const int q = lane4(tid), r4 = (tid & 31) >> 2;
  // fragment row e of this thread: TMEM lane 32 (warp & 3) + 16 hl + r4 + 8 e
  auto frow = [&](int e) { return 32 * (warp & 3) + 16 * hl + r4 + 8 * e; };
  float* const ra = S.ra[wg];
  float* const cb = S.cb[wg];
  float* const cc = S.cc[wg];
  uint8_t* const out = S.out[wg];
  const uint32_t bar_id = 1 + wg;
  int stage = 0;
  uint32_t fph0 = 0u, fph1 = 0u, mph = 0;   // phases of full[wg][0], full[wg][1], mbar
  bool have_r1 = false;                      // first row step sums of this tile ready

  // First row step, partial: thread wt sums the squares of channels 64 h ..
  // 64 h + 63 (h = wt >> 7, one 64-channel box) of row `row` of the tile in
  // shared memory; channel 0, the row mean, is kept apart.
  auto r1_partial = [&](const uint8_t* x) {
    const int h = wt >> 7;
    float2 s2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                    make_float2(0.f, 0.f)};
    float x0 = 0.f;
    const uint8_t* xr = x + h * kBoxBytes + row * 128;
#pragma unroll
    for (int c = 0; c < 8; ++c) {   // 16-byte chunk c of the box: channels 64 h + 8c ..
      uint4 u = *reinterpret_cast<const uint4*>(xr + ((c ^ (row & 7)) << 4));
      if (c == 0 && h == 0) {
        x0 = __half2float(__ushort_as_half((unsigned short)(u.x & 0xFFFFu)));
        u.x &= 0xFFFF0000u;
      }
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
        s2[e] = __ffma2_rn(f, f, s2[e]);
      }
    }
    S.r1part[wg][h][row] = ((s2[0].x + s2[0].y) + (s2[1].x + s2[1].y)) +
                           ((s2[2].x + s2[2].y) + (s2[3].x + s2[3].y));
    if (h == 0) S.r1x0[wg][row] = x0;
  };

  Cand next{a.ntiles, -1, -1};   // load thread: candidate after the tile in flight
  if (load_thread) {
    const int id0 = prepare(fetch_cand(a, blockIdx.x * kWG + wg), 0);
    next = fetch_cand(a, id0 + nw);
  }
  named_sync(bar_id, kWGThreads);

  while (true) {
    const TileInfo cur = S.info[wg][stage];
    if (cur.id >= a.ntiles) break;
    if (stage == 0) {
      wait(&S.full[wg][0], fph0);
      fph0 ^= 1u;
    } else {
      wait(&S.full[wg][1], fph1);
      fph1 ^= 1u;
    }
    uint8_t* const xs = S.x[wg][stage];
    if (mma_thread) {
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
    } else if (load_thread) {
      // the next tile of this pipeline, loading while this one is processed
      // (its stage's last tile finished with it one tile ago); then the
      // metadata of the candidate after it, used one tile from now
      const int id1 = prepare(next, stage ^ 1);
      next = fetch_cand(a, id1 < a.ntiles ? id1 + nw : a.ntiles);
    }
    const int part = cur.part;

    // ---- first row step from X itself: the rotated row y = Hs x / sqrt(128)
    // has mean x_0 / sqrt(128) and variance sum_{k >= 1} x_k^2 / 128 (Hs has
    // orthogonal rows of norm^2 128, and column sums 128, 0, 0, ...); in units
    // of Y = Hs x: mean x_0, variance sum_{k >= 1} x_k^2.  Its sums were taken
    // at the end of the previous tile (the first tile of a pipeline takes
    // them now) ----
    if (!have_r1 && a.iters > 0) {
      r1_partial(xs);
      named_sync(bar_id, kWGThreads);
    }
    if (lower) {
      cb[row] = 1.f;
      cc[row] = 1.f;
      if (a.iters > 0) {
        const float var = S.r1part[wg][0][row] + S.r1part[wg][1][row];
        float sq;
        ra[row] = step_stat(a.rms, S.r1x0[wg][row], var, sq) ? rsqrtf(sq) : kInvSqrt128;
      } else {
        ra[row] = kInvSqrt128;
      }
    }
    named_sync(bar_id, kWGThreads);
    wait(&S.mbar[wg], mph);
    mph ^= 1;
    tc_fence_after();

    // ---- Sinkhorn-like normalization: column step (Y^T: rows = channels),
    // then for the later iterations row step (Y: rows = tokens) and column
    // step.  Each thread holds two rows of each 16-lane half of its warp's
    // lanes, 32 columns of each (16x256b fragments); cb is indexed by Y column
    // (channel chan_of(n)), ra by token ----
    for (int it = 0; it < a.iters; ++it) {
      if (it > 0) {
        float2 w[16];
        frag_weights(cb, q, w);
        float v[64], mean[2], var[2];
        tmem_ld256(tY, v);
        tmem_wait_ld();
        frag_moments(v, w, mean, var);
        if (q == 0) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float sq;
            if (step_stat(a.rms, mean[e], var[e], sq)) ra[frow(e)] = rsqrtf(sq);
          }
        }
        named_sync(bar_id, kWGThreads);
      }
      float2 w[16];
      frag_weights(ra, q, w);
      float v[64], mean[2], var[2];
      tmem_ld256(tYT, v);
      tmem_wait_ld();
      frag_moments(v, w, mean, var);
      if (q == 0) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float sq;
          if (step_stat(a.rms, mean[e], var[e], sq)) {
            const int n = frow(e);
            const float rs = rsqrtf(sq);
            cb[n] = rs;
            cc[chan_of(n)] = sq * rs;
          }
        }
      }
      if (it == a.iters - 1 && leader) bulk_wait_read();
      named_sync(bar_id, kWGThreads);
    }

    // ---- RTN + pack into the staging copy of the record part, written out
    // by one bulk copy; the previous tile's copy has read it by now ----
    if (a.iters == 0) {
      if (leader) bulk_wait_read();
      named_sync(bar_id, kWGThreads);
    }
    const float2 mg = make_float2(kMagic, kMagic);
    if constexpr (RecFmt<FMT>::pc) {
      // per-channel groups: x_td = Y_td / (r_t c_d) = (Y_td ra_t) cb_d, the
      // range of each channel (a row n of Y^T) over the tile's tokens, then
      // the codes: V from the same Y^T fragment, K (token-major) from Y with
      // the channels' minima and 1 / step published in shared memory.  Both
      // passes form x by the same two products, so they see the same values.
      using F = RecFmt<FMT>;
      const float qmax = part ? 3.f : 15.f;
      uint8_t* const meta = out + (part ? F::vc - F::kpart : F::kc);
      float2 wr[16];
      frag_weights(ra, q, wr);
      float v[64];
      tmem_ld256(tYT, v);
      tmem_wait_ld();
      float lo[2], inv[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float cbe = cb[frow(e)];
        const float2 cb2 = make_float2(cbe, cbe);
        float mn = INFINITY, mx = -INFINITY;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float2 x = __fmul2_rn(__fmul2_rn(pair(v, k, e), wr[k]), cb2);
          v[4 * k + 2 * e] = x.x;
          v[4 * k + 2 * e + 1] = x.y;
          mn = min3f(mn, x.x, x.y);
          mx = max3f(mx, x.x, x.y);
        }
        lo[e] = quad_min(mn);
        const float range = quad_max(mx) - lo[e];
        inv[e] = range > 0.f ? __fdividef(qmax, range) : 0.f;
        if (q == 0) {
          const int n = frow(e), ch = chan_of(n);
          S.vmin[wg][n] = lo[e];
          S.vinv[wg][n] = inv[e];
          F::put_bd(meta, ch, cc[ch] * (range / qmax), cc[ch] * lo[e]);
        }
      }
      // r_t = 1 / (ra_t sqrt(128)) in the oracle's units (ra is in units of Y)
      if (lower) F::put_r(out + (part ? F::vsz - F::kpart : F::ksz), row, kInvSqrt128 / ra[row]);
      if (part) {
        // V: whole words of the thread's channels, crumb (k & 7) + 8b of word
        // v_word(channel, q, k >> 3) from token column 8k + 2q + b
        uint32_t* vw = reinterpret_cast<uint32_t*>(out);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float2 nm = make_float2(-lo[e], -lo[e]), iv = make_float2(inv[e], inv[e]);
          uint32_t acc[2] = {0u - kMagicV, 0u - kMagicV};
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float2 f = __ffma2_rn(__fadd2_rn(pair(v, k, e), nm), iv, mg);
            acc[k >> 3] += __float_as_uint(f.x) << (2 * (k & 7));
            acc[k >> 3] += __float_as_uint(f.y) << (2 * (k & 7) + 16);
          }
          *reinterpret_cast<uint2*>(vw + v_word(chan_of(frow(e)), q, 0)) =
              make_uint2(acc[0], acc[1]);
        }
      } else {
        // K: token rows of Y, the channels' minima and 1 / step by column
        named_sync(bar_id, kWGThreads);
        float2 wc[16];
        frag_weights(cb, q, wc);
        tmem_ld256(tY, v);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = frow(e);
          const float2 ra2 = make_float2(ra[t], ra[t]);
          uint32_t acc[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[j] = 0u - kMagicK;
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float2 x = __fmul2_rn(__fmul2_rn(pair(v, k, e), ra2), wc[k]);
            const float2 m2 = *reinterpret_cast<const float2*>(S.vmin[wg] + 8 * k + 2 * q);
            const float2 i2 = *reinterpret_cast<const float2*>(S.vinv[wg] + 8 * k + 2 * q);
            const float2 f =
                __ffma2_rn(__fadd2_rn(x, make_float2(-m2.x, -m2.y)), i2, mg);
            acc[k >> 2] += __float_as_uint(f.x) << (8 * (k & 3));
            acc[k >> 2] += __float_as_uint(f.y) << (8 * (k & 3) + 4);
          }
          *reinterpret_cast<uint4*>(out + kOffKCodes + 64 * t + 16 * q) =
              make_uint4(acc[0], acc[1], acc[2], acc[3]);
        }
      }
    } else {
    float2 w[16];
    frag_weights(cb, q, w);
    float v[64];
    tmem_ld256(tY, v);
    tmem_wait_ld();
    if (part == 0) {
      // K: token-major, 64 bytes per token; nibble e of word w = channel 8w + e.
      // The fragment of a row is the channels 32q .. 32q + 31: its words 4q ..
      // 4q + 3, nibble 2 (k & 3) + b of word 4q + (k >> 2) from column pair k.
      if (lower) RecFmt<FMT>::put_c(out + RecFmt<FMT>::kc, row, cc[row]);
      {
        float mn[2], mx[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          mn[e] = INFINITY;
          mx[e] = -INFINITY;
        }
#pragma unroll
        for (int k = 0; k < 16; ++k)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float2 x = __fmul2_rn(pair(v, k, e), w[k]);
            v[4 * k + 2 * e] = x.x;
            v[4 * k + 2 * e + 1] = x.y;
            mn[e] = min3f(mn[e], x.x, x.y);
            mx[e] = max3f(mx[e], x.x, x.y);
          }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          // the thread's channels 32q .. 32q + 31 lie in group q >> 1 of g64
          constexpr bool G64 = RecFmt<FMT>::g64;
          const float lo = grp_min<G64>(mn[e]), hi = grp_max<G64>(mx[e]);
          const float range = hi - lo;
          constexpr float kq = RecFmt<FMT>::k8 ? 255.f : 15.f;   // 2^bits - 1 of K
          const float inv = range > 0.f ? __fdividef(kq, range) : 0.f;
          const int t = frow(e);
          if ((q & (G64 ? 1 : 3)) == 0)
            RecFmt<FMT>::put_sz_g(out + RecFmt<FMT>::ksz, t, G64 ? q >> 1 : 0,
                                  range * (kInvSqrt128 / kq), lo * kInvSqrt128);
          // u = (x - min) (kq / range) + 1.5 * 2^23: the code in the low bits
          const float2 nm = make_float2(-lo, -lo), iv = make_float2(inv, inv);
          if constexpr (RecFmt<FMT>::k8) {
            // 8-bit: the row's channels 32q .. 32q + 31 are bytes of its
            // chunks 2q, 2q + 1 (swapped in odd tokens): byte 2 (k & 1) + b
            // of word k >> 1 from column pair k
            uint32_t acc[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = 0u - kMagicB;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const float2 f = __ffma2_rn(__fadd2_rn(pair(v, k, e), nm), iv, mg);
              acc[k >> 1] += __float_as_uint(f.x) << (16 * (k & 1));
              acc[k >> 1] += __float_as_uint(f.y) << (16 * (k & 1) + 8);
            }
            uint8_t* const row_out = out + kOffKCodes + 128 * t;
            const int sw = t & 1;
            *reinterpret_cast<uint4*>(row_out + 16 * ((2 * q) ^ sw)) =
                make_uint4(acc[0], acc[1], acc[2], acc[3]);
            *reinterpret_cast<uint4*>(row_out + 16 * ((2 * q + 1) ^ sw)) =
                make_uint4(acc[4], acc[5], acc[6], acc[7]);
          } else {
            uint32_t acc[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[j] = 0u - kMagicK;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const float2 f = __ffma2_rn(__fadd2_rn(pair(v, k, e), nm), iv, mg);
              acc[k >> 2] += __float_as_uint(f.x) << (8 * (k & 3));
              acc[k >> 2] += __float_as_uint(f.y) << (8 * (k & 3) + 4);
            }
            *reinterpret_cast<uint4*>(out + kOffKCodes + 64 * t + 16 * q) =
                make_uint4(acc[0], acc[1], acc[2], acc[3]);
          }
        }
      }
    } else {
      // V: the per-token min and 3 / range from Y, then each thread packs
      // whole words of its channels from Y^T: the fragment columns (tokens)
      // 8k + 2q + b are crumb (k & 7) + 8b of word v_word(channel, q, k >> 3)
      if (lower)
        RecFmt<FMT>::put_c(out + (RecFmt<FMT>::vc - RecFmt<FMT>::kpart), row, cc[row]);
      {
        float mn[2], mx[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          mn[e] = INFINITY;
          mx[e] = -INFINITY;
        }
#pragma unroll
        for (int k = 0; k < 16; ++k)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float2 x = __fmul2_rn(pair(v, k, e), w[k]);
            mn[e] = min3f(mn[e], x.x, x.y);
            mx[e] = max3f(mx[e], x.x, x.y);
          }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          constexpr bool G64 = RecFmt<FMT>::g64;
          const float lo = grp_min<G64>(mn[e]), hi = grp_max<G64>(mx[e]);
          const float range = hi - lo;
          const int t = frow(e);
          if ((q & (G64 ? 1 : 3)) == 0) {
            const int grp = G64 ? q >> 1 : 0;
            S.vmin[wg][grp * kT + t] = lo;
            constexpr float vq = RecFmt<FMT>::v4 ? 15.f : 3.f;   // 2^bits - 1 of V
            S.vinv[wg][grp * kT + t] = range > 0.f ? __fdividef(vq, range) : 0.f;
            RecFmt<FMT>::put_sz_g(out + (RecFmt<FMT>::vsz - RecFmt<FMT>::kpart), t, grp,
                                  range * (kInvSqrt128 / vq), lo * kInvSqrt128);
          }
        }
      }
      named_sync(bar_id, kWGThreads);
      uint32_t* vw = reinterpret_cast<uint32_t*>(out);   // V codes open the V part
      {
        tmem_ld256(tYT, v);
        tmem_wait_ld();
        // 2-bit: 2 words per row, crumb (k & 7) + 8b of word k >> 3; 4-bit:
        // 4 words per row, nibble (k & 3) + 4b of word k >> 2
        constexpr bool V4 = RecFmt<FMT>::v4;
        constexpr int NWV = V4 ? 4 : 2;
        float2 cd2[2];
        uint32_t acc[2][NWV];
        int gofs[2];   // the row's channel group (g64) in the per-token arrays
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float cd = cb[frow(e)];
          cd2[e] = make_float2(cd, cd);
#pragma unroll
          for (int j = 0; j < NWV; ++j) acc[e][j] = 0u - (V4 ? kMagicK : kMagicV);
          gofs[e] = RecFmt<FMT>::g64 ? (chan_of(frow(e)) >> 6) * kT : 0;
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float2 m2 =
                *reinterpret_cast<const float2*>(S.vmin[wg] + gofs[e] + 8 * k + 2 * q);
            const float2 i2 =
                *reinterpret_cast<const float2*>(S.vinv[wg] + gofs[e] + 8 * k + 2 * q);
            const float2 nm = make_float2(-m2.x, -m2.y);
            const float2 d = __ffma2_rn(pair(v, k, e), cd2[e], nm);
            const float2 f = __ffma2_rn(d, i2, mg);
            if constexpr (V4) {
              acc[e][k >> 2] += __float_as_uint(f.x) << (4 * (k & 3));
              acc[e][k >> 2] += __float_as_uint(f.y) << (4 * (k & 3) + 16);
            } else {
              acc[e][k >> 3] += __float_as_uint(f.x) << (2 * (k & 7));
              acc[e][k >> 3] += __float_as_uint(f.y) << (2 * (k & 7) + 16);
            }
          }
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          if constexpr (V4)
            *reinterpret_cast<uint4*>(vw + v4_word(chan_of(frow(e)), q, 0)) =
                make_uint4(acc[e][0], acc[e][1], acc[e][2], acc[e][3]);
          else
            *reinterpret_cast<uint2*>(vw + v_word(chan_of(frow(e)), q, 0)) =
                make_uint2(acc[e][0], acc[e][1]);
        }
      }
    }
    }   // per-token groups
    // the first row step sums of the next tile, whose input is already in the
    // other stage (no MMA reads it yet)
    have_r1 = false;
    if (a.iters > 0) {
      const int nid = S.info[wg][stage ^ 1].id;
      if (nid < a.ntiles) {
        if (stage == 0)
          wait(&S.full[wg][1], fph1);
        else
          wait(&S.full[wg][0], fph0);
        r1_partial(S.x[wg][stage ^ 1]);
        have_r1 = true;
      }
    }
    // the staging copy is complete and TMEM is free for the next tile
    fence_proxy_async_smem();
    tc_fence_before();
    named_sync(bar_id, kWGThreads);
    if (leader && cur.rec >= 0) {
      bulk_s2g(a.pool + cur.rec + (part ? RecFmt<FMT>::kpart : 0), out,
               part ? RecFmt<FMT>::vpart : RecFmt<FMT>::kpart);
      bulk_commit();
    }
    stage ^= 1;
  }
  if (leader) bulk_wait_all();

  // ---- teardown: every MMA was waited for; the packed outputs are written
  // before the CTA's shared memory is released; free TMEM ----
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
  if (a.mode == 0) tail_copy(a, cp);
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
static_assert(kQSmemBytes <= 232448, "one CTA's shared memory is at most 227 KB");

template <int FMT>
cudaError_t launch_tiles(const CUtensorMap& mk, const CUtensorMap& mv, const QTileArgs& qa,
                         const QCopyArgs& cp, cudaStream_t s) {
  static std::atomic<uint64_t> smem_set{0};
  cudaError_t e = ensure_dynamic_smem(quantize_tc_kernel<FMT>, kQSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  const int sms = device_sm_count();
  if (sms <= 0) return cudaErrorNoDevice;
  const int want = (qa.ntiles + kWG - 1) / kWG;
  // one CTA at least: with no tile to quantize it still does the copies
  const int grid = want < 1 ? 1 : want < sms ? want : sms;
  quantize_tc_kernel<FMT><<<grid, kQThreads, kQSmemBytes, s>>>(mk, mv, qa, cp);
  return cudaGetLastError();
}

cudaError_t launch_fmt(int fmt, const CUtensorMap& mk, const CUtensorMap& mv,
                       const QTileArgs& qa, const QCopyArgs& cp, cudaStream_t s) {
  if (fmt == kFmtM16) return launch_tiles<kFmtM16>(mk, mv, qa, cp, s);
  if (fmt == kFmtPC) return launch_tiles<kFmtPC>(mk, mv, qa, cp, s);
  if (fmt == kFmtG64) return launch_tiles<kFmtG64>(mk, mv, qa, cp, s);
  if (fmt == kFmtV4) return launch_tiles<kFmtV4>(mk, mv, qa, cp, s);
  if (fmt == kFmtK8) return launch_tiles<kFmtK8>(mk, mv, qa, cp, s);
  return launch_tiles<kFmtF32>(mk, mv, qa, cp, s);
}

}  // namespace

bool encode_kv_tile_map(CUtensorMap* map, const void* base, int64_t sb, int64_t st, int64_t sh,
                        int batch, int tokens, int hkv, int* roles) {
  return encode_tile_map(map, base, sb, st, sh, batch, tokens, hkv, roles);
}

bool encode_fp16_map_4d(CUtensorMap* map, const void* base, const uint64_t dims[4],
                        const uint64_t strides[3], const uint32_t box[4]) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[4], st[3];
  cuuint32_t bx[4], estr[4] = {1, 1, 1, 1};
  for (int i = 0; i < 4; ++i) {
    d[i] = (cuuint64_t)dims[i];
    bx[i] = (cuuint32_t)box[i];
  }
  for (int i = 0; i < 3; ++i) st[i] = (cuuint64_t)strides[i];
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void*>(base), d, st, bx, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

cudaError_t launch_quantize_blocks(const QuantizeArgs& a, cudaStream_t s) {
  QTileArgs qa{};
  qa.mode = 0;
  qa.batch = a.batch;
  qa.hkv = a.hkv;
  qa.iters = a.iters;
  qa.rms = a.rms;
  qa.nb = a.max_seq / kT;
  qa.ntiles = a.batch * qa.nb * a.hkv * 2;
  qa.seq_lens = a.seq_lens;
  qa.block_table = a.block_table;
  qa.max_blocks = a.max_blocks;
  qa.max_seq = a.max_seq;
  qa.pool = a.pool;
  qa.num_pages = a.num_pages;
  qa.status = a.status;
  QCopyArgs cp{};
  cp.src_k = a.k;
  cp.src_v = a.v;
  cp.sb = a.sb;
  cp.st = a.st;
  cp.sh = a.sh;
  cp.tail_k = a.tail_k;
  cp.tail_v = a.tail_v;
  CUtensorMap mk, mv;
  memset(&mk, 0, sizeof(mk));
  memset(&mv, 0, sizeof(mv));
  if (qa.ntiles > 0) {
    int rk = 0, rv = 0;
    if (!encode_tile_map(&mk, a.k, a.sb, a.st, a.sh, a.batch, a.max_seq, a.hkv, &rk) ||
        !encode_tile_map(&mv, a.v, a.sb, a.st, a.sh, a.batch, a.max_seq, a.hkv, &rv) || rk != rv)
      return cudaErrorInvalidValue;
    qa.roles = rk;
  }
  // the tiles and the leftover-token copies, one launch
  return launch_fmt(a.fmt, mk, mv, qa, cp, s);
}

cudaError_t launch_append_token(const AppendArgs& a, cudaStream_t s) {
  // one launch: every CTA copies the new tokens of its candidate tiles into
  // the tails, and the tails whose block just filled are quantized by the
  // same kernel as the prefill, reading the tail buffers [B][Hkv][128][128]
  QTileArgs qa{};
  qa.mode = 1;
  qa.batch = a.batch;
  qa.hkv = a.hkv;
  qa.iters = a.iters;
  qa.rms = a.rms;
  qa.nb = 1;
  qa.ntiles = a.batch * a.hkv * 2;
  qa.pos = a.pos;
  qa.block_table = a.block_table;
  qa.max_blocks = a.max_blocks;
  qa.max_seq = 0;
  qa.pool = a.pool;
  qa.num_pages = a.num_pages;
  qa.status = a.status;
  QCopyArgs cp{};
  cp.src_k = a.k_new;
  cp.src_v = a.v_new;
  cp.tail_k = a.tail_k;
  cp.tail_v = a.tail_v;
  CUtensorMap mk, mv;
  int rk = 0, rv = 0;
  const int64_t sh = (int64_t)kT * kD, sb = sh * a.hkv;
  if (!encode_tile_map(&mk, a.tail_k, sb, kD, sh, a.batch, kT, a.hkv, &rk) ||
      !encode_tile_map(&mv, a.tail_v, sb, kD, sh, a.batch, kT, a.hkv, &rv))
    return cudaErrorInvalidValue;
  qa.roles = rk;
  return launch_fmt(a.fmt, mk, mv, qa, cp, s);
}

}  // namespace kvarn
