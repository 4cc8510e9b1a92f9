// snapkv.cu -- SnapKV-style one-shot selection of the KV cache at the end of
// prefill: the observation window's attention over the prompt (tensor cores),
// per-position votes, max pooling, top positions per KV head, and the gather
// of the kept tokens into a compact cache.
//
// Method: "Makale Bulteni - SnapKV" (cmlonder.com): the attention of the
// prompt's last 32 or 64 tokens (the observation window) over the earlier
// tokens is scanned once when prefill ends, and each head keeps its most
// critical clustered positions (pooling, then selection); the rest is dropped
// and decode continues on a compact cache of fixed size, each head with its
// own positions.  Readings: vote v_t = the window queries' softmax mass on
// prefix position t, summed over the KV head's query group (softmax over each
// query's causal context, scale as in decode); clustering = 1-D max pooling
// with an odd kernel; the capacity - W largest pooled votes (ties to the
// lower position) and the W window positions are kept, in increasing order.
//
// Scores: CTA = one chunk of 2048 prompt tokens of one (sequence, KV head),
// four row warps (thread r = TMEM lane r = window row r, the rows being the
// window tokens x the group's query heads, 128 per row tile) and one loader
// thread that streams the chunk's K tiles (TMA, 64-channel boxes, 128-byte
// swizzle, two stages) and issues S = Q K^T (tcgen05.mma, M = N = 128,
// K = 128 channels; fp16 q and k multiply exactly, fp32 in TMEM, two S
// buffers).  Two launches: the first takes each row's running maximum and
// sum of 2^(s - m) over its causal keys per chunk; the second merges those
// over the chunks, recomputes S and sums each column's probabilities over the
// rows (a warp transpose-reduce, then the four warps in shared memory) into
// the votes.
#include "kvarn_internal.cuh"
#include "ptx.cuh"

namespace kvarn {
namespace {

using namespace ptx;

constexpr int kSRowWarps = 4;
constexpr int kSThreads = 32 * kSRowWarps + 32;
constexpr int kSProd = 32 * kSRowWarps;            // loader / MMA thread
constexpr uint32_t kSTile = 128 * 128 * 2;
constexpr uint32_t kSBox = kSTile / 2;
constexpr uint32_t kSIdesc = (1u << 4) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
constexpr uint64_t kSWaitNs = 2000000000ull;
constexpr int kSChunk = kSnapChunkTiles * 128;

struct __align__(1024) SSmem {
  uint8_t qa[kSTile];                 // A: window rows [row][channel]
  uint8_t kt[2][kSTile];              // B: K tiles [token][channel], two stages
  float part[kSRowWarps][128];        // a tile's column sums per warp
  float votes[kSChunk];               // this chunk's votes
  uint64_t full[2], kfree[2], sdone[2], sfree[2], qready, drain;
  uint32_t tmem_base;
  int abort;
};
constexpr int kSSmemBytes = (int)sizeof(SSmem) + 1024;

__device__ __forceinline__ float sex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t ssw(int r, int c) {   // 16-byte chunk c of row r
  return (uint32_t)((c >> 3) * kSBox + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__global__ void __launch_bounds__(kSThreads, 1)
    snapkv_scores_kernel(const __grid_constant__ CUtensorMap tm, const SnapArgs a,
                         const int mode) {
  extern __shared__ uint8_t smem_raw[];
  SSmem& S = *reinterpret_cast<SSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~static_cast<uintptr_t>(1023));
  const int chunk = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = a.g;
  int n = a.seq_lens[b];
  if (n < 0 || n > a.max_seq) {
    if (chunk == 0 && kvh == 0 && tid == 0) report(a.status, KVARN_STATUS_BAD_LENGTH);
    n = 0;
  }
  const int npre = n > a.W ? n - a.W : 0;
  const int t0 = chunk * kSChunk;
  // keys of this chunk: every existing token for the statistics, the prefix
  // for the votes
  const int tend = min(t0 + kSChunk, mode == 0 ? n : npre);
  const int ntile = tend > t0 ? (tend - t0 + 127) / 128 : 0;
  float* const st = a.stats + ((int64_t)(b * a.hkv + kvh) * a.nrt * a.nchunks) * 256;
  if (ntile == 0) {
    if (mode == 0) {
      for (int x = tid; x < a.nrt * 128; x += kSThreads) {
        float* e = st + ((int64_t)(x >> 7) * a.nchunks + chunk) * 256 + 2 * (x & 127);
        e[0] = -INFINITY;
        e[1] = 0.f;
      }
    } else {
      float* vo = a.votes + (int64_t)(b * a.hkv + kvh) * a.max_seq;
      for (int x = t0 + tid; x < min(t0 + kSChunk, a.max_seq); x += kSThreads) vo[x] = 0.f;
    }
    return;
  }

  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.kfree[s], 1);
      mbar_init(&S.sdone[s], 1);
      mbar_init(&S.sfree[s], kSRowWarps);
    }
    mbar_init(&S.qready, kSRowWarps);
    mbar_init(&S.drain, 1);
    S.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&S.tmem_base, 256);
    tmem_relinquish();
  }
  for (int x = tid; x < kSChunk; x += kSThreads) S.votes[x] = 0.f;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  auto wait = [&](uint64_t* bar, uint32_t ph) {
    if (*reinterpret_cast<volatile int*>(&S.abort)) return;
    if (!mbar_wait_bounded(bar, ph, kSWaitNs)) {
      *reinterpret_cast<volatile int*>(&S.abort) = 1;
      report(a.status, KVARN_STATUS_TIMEOUT);
    }
  };
  const int total = a.nrt * ntile;   // tiles in issue order: row tile outer

  if (tid == kSProd) {
    // ================= loader and MMA issue =================
    const int rh = a.roles & 3, rtok = (a.roles >> 2) & 3;
    auto load = [&](int jg) {
      const int s = jg & 1, j = jg % ntile;
      if (jg >= 2) wait(&S.kfree[s], ((jg - 2) >> 1) & 1);   // MMA of tile jg - 2 read it
      const int tt = t0 + 128 * j;
      const int c1 = rh == 1 ? kvh : rtok == 1 ? tt : b;
      const int c2 = rh == 2 ? kvh : rtok == 2 ? tt : b;
      const int c3 = rh == 3 ? kvh : rtok == 3 ? tt : b;
      mbar_arrive_expect_tx(&S.full[s], kSTile);
      tma_load_4d(S.kt[s], &tm, 0, c1, c2, c3, &S.full[s]);
      tma_load_4d(S.kt[s] + kSBox, &tm, 64, c1, c2, c3, &S.full[s]);
    };
    load(0);
    for (int jg = 0; jg < total; ++jg) {
      const int s = jg & 1;
      if (jg + 1 < total) load(jg + 1);
      if (jg % ntile == 0) wait(&S.qready, (jg / ntile) & 1);
      wait(&S.full[s], (jg >> 1) & 1);
      if (jg >= 2) wait(&S.sfree[s], ((jg - 2) >> 1) & 1);   // rows read S of tile jg - 2
      tc_fence_after();
      const uint32_t qa = smem_u32(S.qa), ka = smem_u32(S.kt[s]);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = (kk >> 2) * kSBox + (kk & 3) * 32;
        umma_f16(tmem + 128 * s, umma_desc_sw128(qa + off), umma_desc_sw128(ka + off), kSIdesc,
                 kk > 0);
      }
      umma_commit(&S.sdone[s]);
      umma_commit(&S.kfree[s]);
    }
    umma_commit(&S.drain);
    mbar_wait_bounded(&S.drain, 0, kSWaitNs);
    // copies still in flight (a wait gave up) land before the CTA leaves
    for (int jg = total - 2; jg < total; ++jg)
      if (jg >= 0) mbar_wait_bounded(&S.full[jg & 1], (jg >> 1) & 1, kSWaitNs);
  } else if (warp < kSRowWarps) {
    // ================= window rows: thread r = TMEM lane r =================
    const int r = tid;
    const uint32_t tl = tmem + ((uint32_t)(32 * warp) << 16);
    int jg = 0;
    for (int rt = 0; rt < a.nrt; ++rt) {
      const int rg = 128 * rt + r, i = rg / g, hh = rg % g;
      const bool valid = i < a.W;
      const int P = n - a.W + i;                  // this window query's position
      // the window rows of this row tile, fp16 as given (exact products)
      const __half* qrow = a.q + (((int64_t)b * a.W + (valid ? i : 0)) * a.hq + kvh * g + hh) * kD;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const uint4 u = valid ? __ldg(reinterpret_cast<const uint4*>(qrow) + c)
                              : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(S.qa + ssw(r, c)) = u;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.qready);
      // the row's statistics over all chunks (votes), or this chunk's (stats)
      float m = -INFINITY, z = 0.f;
      float* const ste = st + (int64_t)rt * a.nchunks * 256 + 2 * r;
      if (mode == 1) {
        for (int c = 0; c < a.nchunks; ++c) {
          const float mc = ste[(int64_t)c * 256], zc = ste[(int64_t)c * 256 + 1];
          if (mc == -INFINITY) continue;
          const float mn = fmaxf(m, mc);
          z = z * sex2(m - mn) + zc * sex2(mc - mn);
          m = mn;
        }
      }
      const float iz = z > 0.f ? 1.f / z : 0.f;
      for (int j = 0; j < ntile; ++j, ++jg) {
        const int s = jg & 1;
        wait(&S.sdone[s], (jg >> 1) & 1);
        tc_fence_after();
        const int tb = t0 + 128 * j;
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          float v[32];
          tmem_ld32(tl + 128 * s + 32 * c4, v);
          tmem_wait_ld();
          const int tc = tb + 32 * c4;
          if (mode == 0) {
            float mx = -INFINITY;
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const bool vis = valid && tc + k <= P && tc + k < n;
              v[k] = vis ? v[k] * a.scale_log2 : -INFINITY;
              mx = fmaxf(mx, v[k]);
            }
            if (mx != -INFINITY) {
              const float mn = fmaxf(m, mx);
              float acc = 0.f;
#pragma unroll
              for (int k = 0; k < 32; ++k) acc += sex2(v[k] - mn);
              z = z * sex2(m - mn) + acc;
              m = mn;
            }
          } else {
            // probabilities of this row on prefix columns, then the sum of
            // each column over the warp's 32 rows (lane l ends with column l)
#pragma unroll
            for (int k = 0; k < 32; ++k)
              v[k] = valid && tc + k < npre ? sex2(fmaf(v[k], a.scale_log2, -m)) * iz : 0.f;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
              const bool up = (lane & o) != 0;
#pragma unroll
              for (int k = 0; k < o; ++k) {
                const float send = up ? v[k] : v[k + o];
                const float keep = up ? v[k + o] : v[k];
                v[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
              }
            }
            S.part[warp][32 * c4 + lane] = v[0];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.sfree[s]);
        if (mode == 1) {
          named_sync(1, 32 * kSRowWarps);
          S.votes[128 * j + r] += (S.part[0][r] + S.part[1][r]) + (S.part[2][r] + S.part[3][r]);
          named_sync(1, 32 * kSRowWarps);
        }
      }
      if (mode == 0) {
        float* e = st + ((int64_t)rt * a.nchunks + chunk) * 256 + 2 * r;
        e[0] = m;
        e[1] = z;
      }
    }
    if (mode == 1) {
      float* vo = a.votes + (int64_t)(b * a.hkv + kvh) * a.max_seq;
      for (int x = r; x < kSChunk && t0 + x < a.max_seq; x += 32 * kSRowWarps)
        vo[t0 + x] = t0 + x < npre ? S.votes[x] : 0.f;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// ---------------------------------------------------------------- select --

constexpr int kSelThreads = 1024;

__device__ __forceinline__ uint32_t fkey(float x) { return __float_as_uint(x); }   // x >= 0

// inclusive block scan of one int per thread (1024 threads); returns the
// inclusive prefix, *total the block sum
__device__ __forceinline__ int block_scan(int x, int* wsum, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = wsum[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    wsum[lane] = w;
  }
  __syncthreads();
  const int r = x + (warp > 0 ? wsum[warp - 1] : 0);
  *total = wsum[31];
  __syncthreads();
  return r;
}

// CTA per (KV head, sequence): pooled votes, the keep-th largest by a radix
// select on their bit patterns (non-negative floats order as integers), then
// the kept positions in increasing order, ties at the threshold to the lower
// positions, then the window.
__global__ void __launch_bounds__(kSelThreads) snapkv_select_kernel(SnapSelectArgs a) {
  __shared__ int hist[256];
  __shared__ int wsum[32];
  __shared__ uint32_t sh_prefix;
  __shared__ int sh_remaining;
  const int kvh = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  int n = a.seq_lens[b];
  if (n < 0 || n > a.max_seq) n = 0;
  const int npre = n > a.W ? n - a.W : 0;
  const int keep = a.capacity - a.W;
  int32_t* out = a.indices + (int64_t)(b * a.hkv + kvh) * a.capacity;
  if (npre <= keep) {
    for (int j = tid; j < a.capacity; j += kSelThreads) out[j] = j < n ? j : -1;
    return;
  }
  const float* v = a.votes + (int64_t)(b * a.hkv + kvh) * a.max_seq;
  float* pooled = a.pooled + (int64_t)(b * a.hkv + kvh) * a.max_seq;
  const int rad = a.kernel / 2;
  for (int t = tid; t < npre; t += kSelThreads) {
    float mx = v[t];
    for (int d = 1; d <= rad; ++d) {
      if (t - d >= 0) mx = fmaxf(mx, v[t - d]);
      if (t + d < npre) mx = fmaxf(mx, v[t + d]);
    }
    pooled[t] = mx;
  }
  if (tid == 0) {
    sh_prefix = 0u;
    sh_remaining = keep;
  }
  __syncthreads();
  uint32_t mask = 0u;
  for (int shift = 24; shift >= 0; shift -= 8) {
    if (tid < 256) hist[tid] = 0;
    __syncthreads();
    const uint32_t prefix = sh_prefix;
    for (int t = tid; t < npre; t += kSelThreads) {
      const uint32_t key = fkey(pooled[t]);
      if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
    }
    __syncthreads();
    if (tid < 32) {
      // the first bin, from the top, at which the running count reaches
      // `rem`: lane l holds bins 255 - 8l .. 248 - 8l, a warp scan gives the
      // count above each lane's bins, and the one lane whose bins cross `rem`
      // walks them
      const int rem = sh_remaining;
      int c[8], sum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = hist[255 - 8 * tid - i];
        sum += c[i];
      }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += y;
      }
      int cum = incl - sum;
      if (cum < rem && rem <= incl) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (cum + c[i] >= rem) {
            sh_prefix = prefix | ((uint32_t)(255 - 8 * tid - i) << shift);
            sh_remaining = rem - cum;
            break;
          }
          cum += c[i];
        }
      }
    }
    mask |= 255u << shift;
    __syncthreads();
  }
  const uint32_t thr = sh_prefix;      // the keep-th largest key
  const int need_eq = sh_remaining;    // how many keys equal to it are kept
  // compaction in increasing position
  int eq_base = 0, out_base = 0;
  for (int t0 = 0; t0 < npre; t0 += kSelThreads) {
    const int t = t0 + tid;
    const uint32_t key = t < npre ? fkey(pooled[t]) : 0u;
    const bool eq = t < npre && key == thr;
    int eq_tot;
    const int eq_rank = block_scan(eq ? 1 : 0, wsum, &eq_tot) - (eq ? 1 : 0) + eq_base;
    const bool sel = t < npre && (key > thr || (eq && eq_rank < need_eq));
    int sel_tot;
    const int pos = block_scan(sel ? 1 : 0, wsum, &sel_tot) - (sel ? 1 : 0) + out_base;
    if (sel) out[pos] = t;
    eq_base += eq_tot;
    out_base += sel_tot;
  }
  for (int i = tid; i < a.W; i += kSelThreads) out[keep + i] = npre + i;
}

// Kept tokens into the compact cache: grid (ceil(capacity / 32), hkv, batch),
// 8 warps of 4 kept tokens each; lanes 0-15 copy a K row, 16-31 its V row
// (16 bytes each), the four rows' loads issued before their stores.  A
// position outside [0, max_seq) (the -1 padding) gives zeros.
constexpr int kGatherRows = 4;     // kept tokens per warp
constexpr int kGatherWarps = 8;
__global__ void __launch_bounds__(32 * kGatherWarps)
    snapkv_gather_kernel(const __half* __restrict__ k, const __half* __restrict__ v, int64_t sb,
                         int64_t st, int64_t sh, int max_seq, int hkv,
                         const int32_t* __restrict__ idx, int capacity, __half* __restrict__ ko,
                         __half* __restrict__ vo) {
  const int h = blockIdx.y, b = blockIdx.z, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int j0 = (blockIdx.x * kGatherWarps + warp) * kGatherRows;
  const int32_t* irow = idx + ((int64_t)b * hkv + h) * capacity;
  int tl = -1;
  if (lane < kGatherRows && j0 + lane < capacity) tl = irow[j0 + lane];
  const int part = lane >> 4, c = lane & 15;
  const __half* base = (part ? v : k) + (int64_t)b * sb + (int64_t)h * sh;
  uint4 row[kGatherRows];
#pragma unroll
  for (int i = 0; i < kGatherRows; ++i) {
    const int t = __shfl_sync(0xffffffffu, tl, i);
    row[i] = make_uint4(0u, 0u, 0u, 0u);
    if (t >= 0 && t < max_seq)
      row[i] = __ldg(reinterpret_cast<const uint4*>(base + (int64_t)t * st) + c);
  }
#pragma unroll
  for (int i = 0; i < kGatherRows; ++i) {
    const int j = j0 + i;
    if (j >= capacity) break;
    __half* dst = (part ? vo : ko) + (((int64_t)b * capacity + j) * hkv + h) * kD;
    reinterpret_cast<uint4*>(dst)[c] = row[i];
  }
}

}  // namespace

cudaError_t launch_snapkv_scores(const SnapArgs& a, const CUtensorMap& tm, int mode,
                                 cudaStream_t s) {
  static std::atomic<uint64_t> smem_set{0};
  cudaError_t e = ensure_dynamic_smem(snapkv_scores_kernel, kSSmemBytes, smem_set);
  if (e != cudaSuccess) return e;
  dim3 grid(a.nchunks, a.hkv, a.batch);
  snapkv_scores_kernel<<<grid, kSThreads, kSSmemBytes, s>>>(tm, a, mode);
  return cudaGetLastError();
}

cudaError_t launch_snapkv_select(const SnapSelectArgs& a, cudaStream_t s) {
  dim3 grid(a.hkv, a.batch);
  snapkv_select_kernel<<<grid, kSelThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_snapkv_gather(const __half* k, const __half* v, int64_t sb, int64_t st,
                                 int64_t sh, int batch, int max_seq, int hkv,
                                 const int32_t* indices, int capacity, __half* k_out,
                                 __half* v_out, cudaStream_t s) {
  constexpr int per_cta = kGatherWarps * kGatherRows;
  dim3 grid((capacity + per_cta - 1) / per_cta, hkv, batch);
  snapkv_gather_kernel<<<grid, 32 * kGatherWarps, 0, s>>>(k, v, sb, st, sh, max_seq, hkv, indices,
                                                          capacity, k_out, v_out);
  return cudaGetLastError();
}

}  // namespace kvarn
