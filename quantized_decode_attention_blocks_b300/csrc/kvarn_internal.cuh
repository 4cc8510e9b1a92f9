// kvarn_internal.cuh -- layout constants and launcher declarations shared by
// the CUDA translation units of libkvarn.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/kvarn.h"

namespace kvarn {

// Page record layout (one per page and KV head); see include/kvarn.h.
constexpr int kD = 128;           // head_dim = group size
constexpr int kT = 128;           // tokens per page
constexpr int kRec = 15360;       // bytes per record
constexpr int kOffKCodes = 0;     // [128 tokens][64 B]
constexpr int kOffKSZ = 8192;     // [128 tokens]{s', z'} fp32
constexpr int kOffKC = 9216;      // [128 channels] fp32
constexpr int kOffVCodes = 9728;  // [128 channels][32 B]
constexpr int kOffVSZ = 13824;
constexpr int kOffVC = 14848;
constexpr int kKPart = 9728;      // K part: [0, 9728)
constexpr int kVPart = kRec - kKPart;  // V part: [9728, 15360)
// The record formats, all with the codes above: 0 = kvarn_k4v2_g128 (fp32
// metadata, the constants above); 1 = "_m16", s', z' and c_d stored as fp16
// (round to nearest even), 108 B per token-head:
//   [0, 8192) K codes, [8192, 8704) K {s', z'} fp16 pairs, [8704, 8960) K c_d,
//   [8960, 13056) V codes, [13056, 13568) V {s', z'}, [13568, 13824) V c_d;
// 2 = "_pc", one RTN group per channel (over the tile's 128 tokens), the row
// scale r_t stored per token and c_d folded into the per-channel scale and
// zero: yhat_td = r_t (cs_d q_td + cz_d):
//   [0, 8192) K codes, [8192, 8704) K r_t fp32, [8704, 9728) K {cs_d, cz_d}
//   fp32 pairs, [9728, 13824) V codes, [13824, 14336) V r_t, [14336, 15360) V
//   {cs_d, cz_d}.
// 3 = "k4v2_g64", two RTN groups per token (channels 0-63, 64-127), each with
// its own {s', z'} (the row scale folded in):
//   [0, 8192) K codes, [8192, 10240) K {s'_0, z'_0, s'_1, z'_1} fp32 per
//   token, [10240, 10752) K c_d, [10752, 14848) V codes, [14848, 16896) V
//   {s', z'} x 2, [16896, 17408) V c_d.
// 4 = "k4v4_g128", 4-bit values: the K part as in format 0, then V codes
//   [9728, 17920) (2048 words: the code of channel c = 16m + 8e + r, token
//   t = 16k + 8f + 2j + s is nibble 4s + 2(k & 1) + f of word
//   256m + 32r + 8j + 4e + (k >> 1), see v4_word), [17920, 18944) V {s', z'}
//   fp32 per token, [18944, 19456) V c_d.
// 5 = "k8v4_g128", 8-bit keys and 4-bit values: K codes [0, 16384), one byte
//   per channel, token-major, the 16-byte chunks of odd tokens swapped
//   pairwise (channel d of token t at byte 128 t + (d ^ 16 (t & 1)), see
//   k8_byte), [16384, 17408) K {s', z'} fp32 per token, [17408, 17920) K c_d,
//   then the V part of format 4: [17920, 26112) V codes, [26112, 27136) V
//   {s', z'}, [27136, 27648) V c_d.
// Every format dequantizes as yhat_td = alpha_t beta_d q_td + gamma_t delta_d:
// (alpha, gamma) = (s', z') (of d's group for format 3) and beta = delta = c_d
// for formats 0, 1, 3, 4 and 5, alpha = gamma = r_t and (beta, delta) = (cs_d, cz_d)
// for format 2.  The accessors take the address of the field (record part +
// offset).
constexpr int kFmtF32 = 0, kFmtM16 = 1, kFmtPC = 2, kFmtG64 = 3, kFmtV4 = 4, kFmtK8 = 5;
constexpr int kRecMax = 27648;    // the largest record (format 5)
// Byte of the 8-bit K code of channel d, token t (format 5).  In odd tokens
// the 16-byte chunks trade places, so that the eight rows of a decode warp's
// 16-byte loads (two tokens per quarter warp) fall in different banks.
__host__ __device__ constexpr int k8_byte(int d, int t) { return 128 * t + (d ^ (16 * (t & 1))); }
// Word of the 4-bit V code region holding channel c, token-digit j and
// word p = k >> 1 (format 4); its nibble 4s + 2(k & 1) + f holds the token.
__host__ __device__ constexpr int v4_word(int c, int j, int p) {
  return 256 * (c >> 4) + 32 * (c & 7) + 8 * j + 4 * ((c >> 3) & 1) + p;
}
template <int FMT>
struct RecFmt {
  static constexpr bool m16 = FMT == kFmtM16;
  static constexpr bool pc = FMT == kFmtPC;
  static constexpr bool g64 = FMT == kFmtG64;
  static constexpr bool k8 = FMT == kFmtK8;        // 8-bit keys
  static constexpr bool v4 = FMT == kFmtV4 || k8;  // 4-bit values
  static constexpr int bytes = m16 ? 13824 : g64 ? 17408 : k8 ? 27648 : v4 ? 19456 : 15360;
  static constexpr int kpart = m16 ? 8960 : g64 ? 10752 : k8 ? 17920 : 9728;   // K part [0, kpart)
  static constexpr int vpart = bytes - kpart;       // V part [kpart, bytes)
  static constexpr int ksz = k8 ? 16384 : 8192;     // per-token fields
  static constexpr int kc = m16 ? 8704 : pc ? 8704 : g64 ? 10240 : k8 ? 17408 : 9216;   // per-channel
  static constexpr int vsz = m16 ? 13056 : g64 ? 14848 : k8 ? 26112 : v4 ? 17920 : 13824;   // from the start
  static constexpr int vc = m16 ? 13568 : pc ? 14336 : g64 ? 16896 : k8 ? 27136 : v4 ? 18944 : 14848;
  static constexpr int kbits = k8 ? 8 : 4;
  static constexpr int vbits = v4 ? 4 : 2;
  // (alpha_t, gamma_t) of token t for the channels of group g (g = 0 unless
  // g64)
  static __device__ __forceinline__ float2 get_sz_g(const uint8_t* f, int t, int g) {
    if constexpr (g64)
      return reinterpret_cast<const float2*>(f)[2 * t + g];
    else
      return get_sz(f, t);
  }
  static __device__ __forceinline__ void put_sz_g(uint8_t* f, int t, int g, float s, float z) {
    if constexpr (g64)
      reinterpret_cast<float2*>(f)[2 * t + g] = make_float2(s, z);
    else
      put_sz(f, t, s, z);
  }
  // (alpha_t, gamma_t) of token t
  static __device__ __forceinline__ float2 get_sz(const uint8_t* f, int t) {
    static_assert(!g64, "the g64 format has two pairs per token (get_sz_g)");
    if constexpr (m16) {
      return __half22float2(reinterpret_cast<const __half2*>(f)[t]);
    } else if constexpr (pc) {
      const float r = reinterpret_cast<const float*>(f)[t];
      return make_float2(r, r);
    } else {
      return reinterpret_cast<const float2*>(f)[t];
    }
  }
  static __device__ __forceinline__ void put_sz(uint8_t* f, int t, float s, float z) {
    static_assert(!pc, "the per-channel format stores r_t (put_r)");
    static_assert(!g64, "the g64 format has two pairs per token (put_sz_g)");
    if constexpr (m16)
      reinterpret_cast<__half2*>(f)[t] = __floats2half2_rn(s, z);
    else
      reinterpret_cast<float2*>(f)[t] = make_float2(s, z);
  }
  static __device__ __forceinline__ void put_r(uint8_t* f, int t, float r) {
    static_assert(pc, "only the per-channel format stores r_t");
    reinterpret_cast<float*>(f)[t] = r;
  }
  // (beta_d, delta_d) of channel d
  static __device__ __forceinline__ float2 get_bd(const uint8_t* f, int d) {
    if constexpr (pc) {
      return reinterpret_cast<const float2*>(f)[d];
    } else {
      const float c = m16 ? __half2float(reinterpret_cast<const __half*>(f)[d])
                          : reinterpret_cast<const float*>(f)[d];
      return make_float2(c, c);
    }
  }
  // beta of channels 4 i .. 4 i + 3, and delta of the same channels
  static __device__ __forceinline__ float4 get_b4(const uint8_t* f, int i) {
    if constexpr (m16) {
      const uint2 u = reinterpret_cast<const uint2*>(f)[i];
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
      const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
      return make_float4(a.x, a.y, b.x, b.y);
    } else if constexpr (pc) {
      const float4 p0 = reinterpret_cast<const float4*>(f)[2 * i];
      const float4 p1 = reinterpret_cast<const float4*>(f)[2 * i + 1];
      return make_float4(p0.x, p0.z, p1.x, p1.z);
    } else {
      return reinterpret_cast<const float4*>(f)[i];
    }
  }
  static __device__ __forceinline__ float4 get_d4(const uint8_t* f, int i) {
    if constexpr (pc) {
      const float4 p0 = reinterpret_cast<const float4*>(f)[2 * i];
      const float4 p1 = reinterpret_cast<const float4*>(f)[2 * i + 1];
      return make_float4(p0.y, p0.w, p1.y, p1.w);
    } else {
      return get_b4(f, i);
    }
  }
  static __device__ __forceinline__ void put_c(uint8_t* f, int d, float c) {
    static_assert(!pc, "the per-channel format stores {cs, cz} (put_bd)");
    if constexpr (m16)
      reinterpret_cast<__half*>(f)[d] = __float2half_rn(c);
    else
      reinterpret_cast<float*>(f)[d] = c;
  }
  static __device__ __forceinline__ void put_bd(uint8_t* f, int d, float cs, float cz) {
    static_assert(pc, "only the per-channel format stores {cs, cz}");
    reinterpret_cast<float2*>(f)[d] = make_float2(cs, cz);
  }
};
static_assert(RecFmt<kFmtF32>::bytes == kRec && RecFmt<kFmtF32>::kpart == kKPart &&
                  RecFmt<kFmtF32>::ksz == kOffKSZ && RecFmt<kFmtF32>::kc == kOffKC &&
                  RecFmt<kFmtF32>::vsz == kOffVSZ && RecFmt<kFmtF32>::vc == kOffVC &&
                  RecFmt<kFmtF32>::kpart == kOffVCodes,
              "the fp32 format is the one the constants above describe");
static_assert(RecFmt<kFmtM16>::kpart % 16 == 0 && RecFmt<kFmtM16>::vpart % 16 == 0 &&
                  RecFmt<kFmtM16>::bytes % 16 == 0 && RecFmt<kFmtM16>::vsz % 16 == 0 &&
                  RecFmt<kFmtM16>::vc % 16 == 0 && RecFmt<kFmtM16>::kc % 16 == 0 &&
                  RecFmt<kFmtPC>::kc % 16 == 0 && RecFmt<kFmtPC>::vc % 16 == 0 &&
                  RecFmt<kFmtG64>::kpart % 16 == 0 && RecFmt<kFmtG64>::vpart % 16 == 0 &&
                  RecFmt<kFmtG64>::kc % 16 == 0 && RecFmt<kFmtG64>::vsz % 16 == 0 &&
                  RecFmt<kFmtG64>::vc % 16 == 0 && RecFmt<kFmtV4>::vsz % 16 == 0 &&
                  RecFmt<kFmtV4>::vc % 16 == 0 && RecFmt<kFmtK8>::kpart % 16 == 0 &&
                  RecFmt<kFmtK8>::vsz % 16 == 0 && RecFmt<kFmtK8>::vc % 16 == 0 &&
                  RecFmt<kFmtK8>::kc % 16 == 0 && RecFmt<kFmtK8>::vpart == RecFmt<kFmtV4>::vpart &&
                  RecFmt<kFmtK8>::bytes == kRecMax,
              "bulk copies and vector loads need 16-byte parts and fields");
// The format code of a configuration.
__host__ __device__ constexpr int fmt_of(int meta16, int per_channel, int group, int v_bits,
                                         int k_bits = 4) {
  return k_bits == 8 ? kFmtK8 : v_bits == 4 ? kFmtV4 : group == 64 ? kFmtG64
         : per_channel ? kFmtPC : meta16 ? kFmtM16 : kFmtF32;
}
inline int cfg_fmt(const kvarn_config_t* c) {
  return fmt_of(c->meta_fp16, c->per_channel, c->group, c->v_bits, c->k_bits);
}

// Split-K partial state per (sequence, query head, split): m, l, 2 pad, o[128]
// (o 16-byte aligned).
constexpr int kPartStride = 4 + kD;

// V codes: 2 bits each, 1024 little-endian 32-bit words.  With channel
// c = 16m + 8e + r and token t = 16k + 8f + 2j + s, the code of (c, t) is crumb
// 2(k & 3) + f + 8s of word 128m + 16r + 4j + 2e + (k >> 2).  One lane of a
// decode warp (lane = 4r + j) then finds all the codes it feeds to the tensor
// cores for channels 16m + r and 16m + 8 + r in four consecutive words.
__host__ __device__ constexpr int v_word(int c, int j, int h) {
  return 128 * (c >> 4) + 16 * (c & 7) + 4 * j + 2 * ((c >> 3) & 1) + h;
}
// token held by crumb i (0..15) of the words (j, h) of any channel
__host__ __device__ constexpr int v_token(int j, int h, int i) {
  return 16 * (4 * h + ((i & 7) >> 1)) + 8 * (i & 1) + 2 * j + (i >> 3);
}
constexpr int kMaxG = 16;         // query heads per KV head supported
constexpr int kMaxIters = 64;     // Sinkhorn iterations accepted

// Streaming multiprocessors of the current device, queried once per device
// (cudaDevAttrMultiProcessorCount) and cached; 0 when no device answers.
// Grids and split plans are sized from it, so they follow the actual chip.
int device_sm_count();

// 1 / sqrt(128), rounded to fp32.
constexpr float kInvSqrt128 = 0.08838834764831845f;

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current
// device.  cudaFuncSetAttribute acts on the current device only, so `done`
// keeps one bit per device id (0-63) where it has been applied; other ids
// apply it on every call.  Safe to call from several host threads, and after
// the first call on a device it makes no CUDA call besides cudaGetDevice (so
// it may run inside a stream capture).
template <typename Kernel>
cudaError_t ensure_dynamic_smem(Kernel* kernel, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
  return e;
}

struct QuantizeArgs {
  const __half* k;
  const __half* v;
  int64_t sb, st, sh;       // element strides of k / v
  int batch, hkv, iters, max_seq;
  int rms;                  // Sinkhorn statistic: 0 centred std, 1 uncentred RMS
  int fmt;                  // record format (kFmtF32, kFmtM16, kFmtPC)
  const int32_t* seq_lens;
  const int32_t* block_table;
  int max_blocks;
  uint8_t* pool;
  int64_t num_pages;
  __half* tail_k;
  __half* tail_v;
  int32_t* status;
};

struct AppendArgs {
  const __half* k_new;
  const __half* v_new;
  const int32_t* pos;
  int batch, hkv, iters;
  int rms;
  int fmt;                  // record format
  const int32_t* block_table;
  int max_blocks;
  uint8_t* pool;
  int64_t num_pages;
  __half* tail_k;
  __half* tail_v;
  int32_t* status;
};

struct DecodeArgs {
  const __half* q;
  const uint8_t* pool;
  int64_t num_pages;
  const int32_t* block_table;
  int max_blocks;
  const int32_t* seq_lens;
  int batch, max_seq, hq, hkv, g;
  const __half* tail_k;
  const __half* tail_v;
  float scale;
  __half* out;
  float* ws_part;     // [batch][hq][nsplit][2 + 128]: m, l, o[128]
  int* ws_count;      // [batch][hkv] arrival tickets, zero between calls
  int pages_per_split;
  int nsplit;
  int cluster;        // 1: the nsplit CTAs of a (sequence, KV head) form a cluster
  int fmt;            // record format (kFmtF32, kFmtM16, kFmtPC)
  int32_t* status;
};

// Split-K plan for decode: pages per CTA and the number of splits, both a
// pure function of (batch, hkv, max_seq) so that the workspace query and the
// launch agree.
struct DecodePlan {
  int pages_per_split;
  int nsplit;
  bool cluster;        // splits merged inside a thread-block cluster (no tickets read)
  size_t part_bytes;   // partial-state region
  size_t count_bytes;  // ticket region
};
// `num_sms`: streaming multiprocessors the plan fills (device_sm_count()).
// `fmt`: the record format, which sets the kernel's shared memory per CTA.
DecodePlan decode_plan(int batch, int hq, int hkv, int max_seq, int num_sms, int fmt);

cudaError_t launch_quantize_blocks(const QuantizeArgs& a, cudaStream_t s);
cudaError_t launch_append_token(const AppendArgs& a, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_dequantize(int fmt, const uint8_t* rec, int64_t n, float* yk, float* yv,
                              cudaStream_t s);

// A 4-D tensor map over fp16 data with 128-byte swizzle (dims and box
// innermost first, strides of dimensions 1..3 in bytes); false if the driver
// rejects it.
bool encode_fp16_map_4d(CUtensorMap* map, const void* base, const uint64_t dims[4],
                        const uint64_t strides[3], const uint32_t box[4]);

// Tensor map over fp16 [B][S][Hkv][128] (element strides sb, st, sh) with
// boxes of 64 channels x 128 tokens of one (head, sequence), 128-byte swizzle;
// the three outer dimensions ordered by stride, *roles = the map dimension of
// the head (bits 0-1) and of the token (bits 2-3).  False if the driver
// rejects it.
bool encode_kv_tile_map(CUtensorMap* map, const void* base, int64_t sb, int64_t st, int64_t sh,
                        int batch, int tokens, int hkv, int* roles);

// SnapKV-style selection: scores of the observation window over the prefix.
struct SnapArgs {
  const __half* q;            // [B][W][Hq][128] window queries
  int W;                      // window tokens
  int batch, max_seq, hq, hkv, g;
  int roles;                  // tensor-map dimensions of (head, token) for k
  const int32_t* seq_lens;    // prompt lengths n (window included)
  float scale_log2;           // softmax scale * log2(e)
  int nrt;                    // 128-row tiles of the W x g window rows
  int nchunks;                // token chunks per sequence
  float* stats;               // [B][Hkv][nrt][nchunks][128]{m, Z} (workspace)
  float* votes;               // [B][Hkv][max_seq]
  int32_t* status;
};
constexpr int kSnapChunkTiles = 16;   // 2048 tokens per CTA
cudaError_t launch_snapkv_scores(const SnapArgs& a, const CUtensorMap& tm, int mode,
                                 cudaStream_t s);
struct SnapSelectArgs {
  const float* votes;         // [B][Hkv][max_seq]
  float* pooled;              // [B][Hkv][max_seq] (workspace)
  const int32_t* seq_lens;
  int batch, hkv, max_seq, W, capacity, kernel;
  int32_t* indices;           // [B][Hkv][capacity]
};
cudaError_t launch_snapkv_select(const SnapSelectArgs& a, cudaStream_t s);
cudaError_t launch_snapkv_gather(const __half* k, const __half* v, int64_t sb, int64_t st,
                                 int64_t sh, int batch, int max_seq, int hkv,
                                 const int32_t* indices, int capacity, __half* k_out,
                                 __half* v_out, cudaStream_t s);

// The FP16 paged cache the quantized one is compared with.
constexpr int kF16PageBytes = 2 * kT * kD * 2;   // K then V, [128 tokens][128] fp16 each

struct F16WriteArgs {
  const __half* k;
  const __half* v;
  int64_t sb, st, sh;
  int batch, hkv, max_seq;
  const int32_t* seq_lens;
  const int32_t* block_table;
  int max_blocks;
  uint8_t* pool;
  int64_t num_pages;
  int32_t* status;
};

struct F16DecodeArgs {
  const __half* q;
  int64_t num_pages;
  const int32_t* block_table;
  int max_blocks;
  const int32_t* seq_lens;
  int batch, max_seq, hq, hkv, g;
  float scale;
  __half* out;
  float* ws_part;     // [batch][hq][nsplit][kPartStride]
  int* ws_count;      // [batch][hkv] arrival tickets, zero between calls
  int pages_per_split;
  int nsplit;
  int32_t* status;
};
DecodePlan fp16_decode_plan(int batch, int hq, int hkv, int max_seq, int num_sms);
cudaError_t launch_fp16_write(const F16WriteArgs& a, cudaStream_t s);
cudaError_t launch_fp16_decode(const F16DecodeArgs& a, const void* pool, cudaStream_t s);
// The FP8 paged cache (same argument records; pages of KVARN_FP8_PAGE_BYTES).
DecodePlan fp8_decode_plan(int batch, int hq, int hkv, int max_seq, int num_sms);
cudaError_t launch_fp8_write(const F16WriteArgs& a, cudaStream_t s);
cudaError_t launch_fp8_decode(const F16DecodeArgs& a, const void* pool, cudaStream_t s);

// Chunked prefill: attention of a chunk of query tokens over the quantized cache.
struct ChunkArgs {
  const __half* q;            // [batch][M][hq][128]
  int M;                      // query tokens per sequence in q / out
  const int32_t* start;       // [batch] tokens before the chunk
  const int32_t* chunk_lens;  // [batch] query tokens of the chunk (<= M)
  int batch, max_seq, hq, hkv, g;
  int tq;                     // query tokens per 128-row tile (128 / g)
  int ntq;                    // tiles per sequence, ceil(M / tq)
  const uint8_t* pool;
  int64_t num_pages;
  const int32_t* block_table;
  int max_blocks;
  const __half* tail_k;
  const __half* tail_v;
  float scale_log2;           // softmax scale * log2(e)
  __half* out;                // [batch][M][hq][128]
  int fmt;                    // record format (kFmtF32, kFmtM16, kFmtPC)
  int32_t* status;
};
int chunk_rows_per_tile(int g);
cudaError_t launch_chunk_attention(const ChunkArgs& a, cudaStream_t s);

cudaError_t launch_wait_check(int32_t* status, uint64_t limit_ns, int arrive, cudaStream_t s);

__device__ __forceinline__ void report(int32_t* status, int bits) {
  if (status) atomicOr(status, bits);
}

}  // namespace kvarn
