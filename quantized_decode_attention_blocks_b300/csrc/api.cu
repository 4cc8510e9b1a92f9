// api.cu -- the extern "C" boundary of libkvarn (declared in include/kvarn.h):
// argument validation on the host, the split-K plan, launch dispatch.
// Nothing here allocates memory or keeps state between calls.
#include <string.h>

#include "kvarn_internal.cuh"

namespace kvarn {

cudaError_t launch_decode_simple(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_mma(const DecodeArgs& a, cudaStream_t s);
bool decode_mma_supported(int g);
int decode_mma_ctas_per_sm(int g, int fmt);
int decode_mma_resident_per_sm(int g, int fmt);
int decode_simple_ctas_per_sm();
int decode_mma_warps();
int decode_mma_max_cluster();

static inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int device_sm_count() {
  // one slot per device id 0-63; other ids query every time
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 0;
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

// A grid with more (sequence, KV head) groups than resident CTAs runs in
// several waves, balanced by the hardware scheduler; there the plan cuts long
// sequences into runs of at most this many pages, so that no long run keeps
// its SM busy after the rest of the grid is done (mixed serving, 128 lengths
// in [1K, 32K], one CTA per group: 490 us; runs of 32-48 pages: 418 us).
constexpr int64_t kWavePages = 32;

DecodePlan decode_plan(int batch, int hq, int hkv, int max_seq, int num_sms, int fmt) {
  DecodePlan p{};
  // Work unit = one page of one (sequence, KV head); the fp16 tail rides with
  // the split that holds the last page.  The number of splits per (sequence,
  // KV head) is the largest that keeps the whole grid resident at once (one
  // wave, no straggling second wave), but no more than gives every warp of a
  // tensor-core CTA (or two pages of a CUDA-core CTA) something to do.
  const int g = hq / hkv;
  const bool mma = decode_mma_supported(g);
  const int64_t units = max_seq / kT > 0 ? (int64_t)max_seq / kT : 1;
  const int64_t groups = (int64_t)batch * hkv;
  const int64_t slots = (int64_t)(num_sms > 0 ? num_sms : 1) *
                        (mma ? decode_mma_ctas_per_sm(g, fmt) : decode_simple_ctas_per_sm());
  const int64_t min_pages = mma ? decode_mma_warps() : 2;
  int64_t ns = slots / groups;
  const int64_t ns_cap = (units + min_pages - 1) / min_pages;
  if (ns > ns_cap) ns = ns_cap;
  if (ns < 1) ns = 1;
  // Several waves (tensor-core kernel; the pairs alone outnumber the CTAs
  // that can be resident, e.g. three per SM for one head tile): runs of at
  // most kWavePages pages, as many as keep the partial states within the
  // no-alloc scratch; these splits merge through the workspace, since a
  // cluster whose CTAs hold runs of very different lengths keeps its slots
  // busy for the longest.  (48 x 8 pairs of 8K tokens fit one wave of three
  // per SM: split in two they decode in 88 us instead of 82.)
  const bool waves =
      mma && groups > (int64_t)(num_sms > 0 ? num_sms : 1) * decode_mma_resident_per_sm(g, fmt);
  if (waves) {
    const int64_t per_split = groups * g * kPartStride * (int64_t)sizeof(float);
    const int64_t counts = (groups * (int64_t)sizeof(int) + 255) & ~(int64_t)255;
    const int64_t room = ((int64_t)KVARN_NOALLOC_SCRATCH_BYTES - counts - 256) / per_split;
    const int64_t want = (units + kWavePages - 1) / kWavePages;
    ns = want < room ? want : room;
    if (ns < 1) ns = 1;
  }
  const int64_t pps = (units + ns - 1) / ns;
  p.pages_per_split = (int)pps;
  p.nsplit = (int)((units + pps - 1) / pps);
  p.cluster = mma && !waves && p.nsplit >= 2 && p.nsplit <= decode_mma_max_cluster();
  if (p.nsplit > 1) {
    p.part_bytes = (size_t)batch * hq * p.nsplit * kPartStride * sizeof(float);
    p.part_bytes = (p.part_bytes + 255) & ~(size_t)255;
    p.count_bytes = ((size_t)batch * hkv * sizeof(int) + 255) & ~(size_t)255;
  }
  return p;
}

}  // namespace kvarn

using namespace kvarn;

extern "C" {

int kvarn_config_validate(const kvarn_config_t* c) {
  if (!c) return KVARN_ERR_INVALID_ARG;
  if (c->num_q_heads <= 0 || c->num_kv_heads <= 0 || c->num_q_heads % c->num_kv_heads)
    return KVARN_ERR_INVALID_ARG;
  if (c->num_q_heads / c->num_kv_heads > kMaxG) return KVARN_ERR_UNSUPPORTED;
  if (c->head_dim != kD || c->block_tokens != kT || (c->group != kD && c->group != 64) ||
      (c->k_bits != 4 && c->k_bits != 8) || (c->v_bits != 2 && c->v_bits != 4))
    return KVARN_ERR_UNSUPPORTED;
  if (c->sinkhorn_iters < 0 || c->sinkhorn_iters > kMaxIters) return KVARN_ERR_UNSUPPORTED;
  if (c->sinkhorn_rms != 0 && c->sinkhorn_rms != 1) return KVARN_ERR_UNSUPPORTED;
  if (c->meta_fp16 != 0 && c->meta_fp16 != 1) return KVARN_ERR_UNSUPPORTED;
  if (c->per_channel != 0 && c->per_channel != 1) return KVARN_ERR_UNSUPPORTED;
  if (c->per_channel && c->meta_fp16) return KVARN_ERR_UNSUPPORTED;   // fp32 metadata only
  if (c->group == 64 && (c->per_channel || c->meta_fp16)) return KVARN_ERR_UNSUPPORTED;
  if (c->v_bits == 4 && (c->group != kD || c->per_channel || c->meta_fp16))
    return KVARN_ERR_UNSUPPORTED;
  if (c->k_bits == 8 && c->v_bits != 4) return KVARN_ERR_UNSUPPORTED;   // "k8v4_g128" only
  return KVARN_OK;
}

int kvarn_config_from_string(const char* s, int hq, int hkv, kvarn_config_t* out) {
  if (!s || !out) return KVARN_ERR_INVALID_ARG;
  if (!strncmp(s, "kvarn_", 6)) s += 6;
  int group, kbits = 4, vbits = 2;
  const char* rest;
  if (!strncmp(s, "k4v2_g128", 9)) {
    group = kD;
    rest = s + 9;
  } else if (!strncmp(s, "k4v2_g64", 8)) {
    group = 64;
    rest = s + 8;
  } else if (!strncmp(s, "k4v4_g128", 9)) {
    group = kD;
    vbits = 4;
    rest = s + 9;
  } else if (!strncmp(s, "k8v4_g128", 9)) {
    group = kD;
    kbits = 8;
    vbits = 4;
    rest = s + 9;
  } else {
    return KVARN_ERR_UNSUPPORTED;
  }
  int iters = 2, rms = 0, m16 = 0, pc = 0;
  // the variant suffixes, each at most once and in either order, then "_s<K>"
  for (;;) {
    if (!rms && !strncmp(rest, "_rms", 4)) {
      rms = 1;
      rest += 4;
    } else if (!m16 && !strncmp(rest, "_m16", 4)) {
      m16 = 1;
      rest += 4;
    } else if (!pc && !strncmp(rest, "_pc", 3) && (rest[3] == 0 || rest[3] == '_')) {
      pc = 1;
      rest += 3;
    } else {
      break;
    }
  }
  if (*rest) {
    if (rest[0] != '_' || rest[1] != 's' || !rest[2]) return KVARN_ERR_UNSUPPORTED;
    int v = 0;
    for (const char* p = rest + 2; *p; ++p) {
      if (*p < '0' || *p > '9' || v > kMaxIters) return KVARN_ERR_UNSUPPORTED;
      v = v * 10 + (*p - '0');
    }
    iters = v;
  }
  kvarn_config_t c;
  c.head_dim = kD;
  c.block_tokens = kT;
  c.group = group;
  c.k_bits = kbits;
  c.v_bits = vbits;
  c.sinkhorn_iters = iters;
  c.sinkhorn_rms = rms;
  c.meta_fp16 = m16;
  c.per_channel = pc;
  c.num_q_heads = hq;
  c.num_kv_heads = hkv;
  const int rc = kvarn_config_validate(&c);
  if (rc != KVARN_OK) return rc;
  *out = c;
  return KVARN_OK;
}

size_t kvarn_page_bytes(const kvarn_config_t* c) {
  if (kvarn_config_validate(c) != KVARN_OK) return 0;
  if (c->group == 64) return (size_t)RecFmt<kFmtG64>::bytes;
  if (c->k_bits == 8) return (size_t)RecFmt<kFmtK8>::bytes;
  if (c->v_bits == 4) return (size_t)RecFmt<kFmtV4>::bytes;
  return c->meta_fp16 ? (size_t)RecFmt<kFmtM16>::bytes : (size_t)RecFmt<kFmtF32>::bytes;
}

int kvarn_quantize_blocks(const kvarn_config_t* cfg, const void* k, const void* v,
                          int64_t stride_b, int64_t stride_t, int64_t stride_h, int batch,
                          const int32_t* seq_lens, int max_seq, const int32_t* block_table,
                          int max_blocks, void* pool, int64_t num_pages, void* tail_k,
                          void* tail_v, int32_t* status, kvarn_stream_t stream) {
  int rc = kvarn_config_validate(cfg);
  if (rc != KVARN_OK) return rc;
  if (batch < 0 || max_seq < 0 || max_blocks < 0 || num_pages < 0) return KVARN_ERR_INVALID_ARG;
  if (batch == 0 || max_seq == 0) return KVARN_OK;
  if (!k || !v || !seq_lens || !tail_k || !tail_v) return KVARN_ERR_INVALID_ARG;
  if (max_seq >= kT && (!block_table || !pool || num_pages <= 0)) return KVARN_ERR_INVALID_ARG;
  if ((int64_t)max_blocks * kT < (int64_t)(max_seq / kT) * kT) return KVARN_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(pool) || !aligned16(tail_k) ||
      !aligned16(tail_v))
    return KVARN_ERR_INVALID_ARG;
  if (stride_b < 0 || stride_t < kD || stride_h < kD || (stride_b | stride_t | stride_h) % 8)
    return KVARN_ERR_INVALID_ARG;
  if ((int64_t)max_seq / kT + 1 > 65535 || 2 * cfg->num_kv_heads > 65535 || batch > 65535)
    return KVARN_ERR_UNSUPPORTED;
  QuantizeArgs a;
  a.k = static_cast<const __half*>(k);
  a.v = static_cast<const __half*>(v);
  a.sb = stride_b;
  a.st = stride_t;
  a.sh = stride_h;
  a.batch = batch;
  a.hkv = cfg->num_kv_heads;
  a.iters = cfg->sinkhorn_iters;
  a.rms = cfg->sinkhorn_rms;
  a.fmt = cfg_fmt(cfg);
  a.max_seq = max_seq;
  a.seq_lens = seq_lens;
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.pool = static_cast<uint8_t*>(pool);
  a.num_pages = num_pages;
  a.tail_k = static_cast<__half*>(tail_k);
  a.tail_v = static_cast<__half*>(tail_v);
  a.status = status;
  return launch_quantize_blocks(a, (cudaStream_t)stream) == cudaSuccess ? KVARN_OK
                                                                         : KVARN_ERR_LAUNCH;
}

int kvarn_append_token(const kvarn_config_t* cfg, const void* k_new, const void* v_new,
                       const int32_t* pos, int batch, const int32_t* block_table,
                       int max_blocks, void* pool, int64_t num_pages, void* tail_k,
                       void* tail_v, int32_t* status, kvarn_stream_t stream) {
  int rc = kvarn_config_validate(cfg);
  if (rc != KVARN_OK) return rc;
  if (batch < 0 || max_blocks < 0 || num_pages < 0) return KVARN_ERR_INVALID_ARG;
  if (batch == 0) return KVARN_OK;
  if (!k_new || !v_new || !pos || !block_table || !pool || !tail_k || !tail_v ||
      max_blocks == 0 || num_pages == 0)
    return KVARN_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(pool) || !aligned16(tail_k) ||
      !aligned16(tail_v))
    return KVARN_ERR_INVALID_ARG;
  if (batch > 65535) return KVARN_ERR_UNSUPPORTED;
  AppendArgs a;
  a.k_new = static_cast<const __half*>(k_new);
  a.v_new = static_cast<const __half*>(v_new);
  a.pos = pos;
  a.batch = batch;
  a.hkv = cfg->num_kv_heads;
  a.iters = cfg->sinkhorn_iters;
  a.rms = cfg->sinkhorn_rms;
  a.fmt = cfg_fmt(cfg);
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.pool = static_cast<uint8_t*>(pool);
  a.num_pages = num_pages;
  a.tail_k = static_cast<__half*>(tail_k);
  a.tail_v = static_cast<__half*>(tail_v);
  a.status = status;
  return launch_append_token(a, (cudaStream_t)stream) == cudaSuccess ? KVARN_OK
                                                                      : KVARN_ERR_LAUNCH;
}

int kvarn_decode_split_plan(const kvarn_config_t* cfg, int batch, int max_seq, int num_sms,
                            int* pages_per_split, int* nsplit, size_t* workspace_bytes) {
  const int rc = kvarn_config_validate(cfg);
  if (rc != KVARN_OK) return rc;
  if (batch <= 0 || max_seq < 0) return KVARN_ERR_INVALID_ARG;
  if (num_sms <= 0) {
    num_sms = device_sm_count();
    if (num_sms <= 0) return KVARN_ERR_LAUNCH;
  }
  const DecodePlan p =
      decode_plan(batch, cfg->num_q_heads, cfg->num_kv_heads, max_seq, num_sms, cfg_fmt(cfg));
  if (pages_per_split) *pages_per_split = p.pages_per_split;
  if (nsplit) *nsplit = p.nsplit;
  if (workspace_bytes) *workspace_bytes = p.part_bytes + p.count_bytes;
  return KVARN_OK;
}

size_t kvarn_decode_workspace_bytes(const kvarn_config_t* cfg, int batch, int max_seq) {
  size_t bytes = 0;
  if (kvarn_decode_split_plan(cfg, batch, max_seq, 0, nullptr, nullptr, &bytes) != KVARN_OK)
    return 0;
  return bytes;
}

int kvarn_decode_attention(const kvarn_config_t* cfg, const void* q, const void* pool,
                           int64_t num_pages, const int32_t* block_table, int max_blocks,
                           const int32_t* seq_lens, int batch, int max_seq, const void* tail_k,
                           const void* tail_v, float softmax_scale, void* out, void* workspace,
                           size_t workspace_bytes, int32_t* status, kvarn_stream_t stream) {
  int rc = kvarn_config_validate(cfg);
  if (rc != KVARN_OK) return rc;
  if (batch < 0 || max_seq < 0 || max_blocks < 0 || num_pages < 0) return KVARN_ERR_INVALID_ARG;
  if (batch == 0) return KVARN_OK;
  if (!q || !seq_lens || !tail_k || !tail_v || !out) return KVARN_ERR_INVALID_ARG;
  if (max_seq >= kT && (!pool || !block_table || num_pages <= 0 || max_blocks < max_seq / kT))
    return KVARN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(pool) || !aligned16(tail_k) || !aligned16(tail_v) ||
      !aligned16(out) || !aligned16(workspace))
    return KVARN_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || softmax_scale != softmax_scale) return KVARN_ERR_INVALID_ARG;
  if (batch > 65535 || cfg->num_kv_heads > 65535) return KVARN_ERR_UNSUPPORTED;
  const int sms = device_sm_count();
  if (sms <= 0) return KVARN_ERR_LAUNCH;
  const DecodePlan p =
      decode_plan(batch, cfg->num_q_heads, cfg->num_kv_heads, max_seq, sms, cfg_fmt(cfg));
  if (p.nsplit > 1 && (!workspace || workspace_bytes < p.part_bytes + p.count_bytes))
    return KVARN_ERR_WORKSPACE;
  DecodeArgs a;
  a.q = static_cast<const __half*>(q);
  a.pool = static_cast<const uint8_t*>(pool);
  a.num_pages = num_pages;
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.seq_lens = seq_lens;
  a.batch = batch;
  a.max_seq = max_seq;
  a.hq = cfg->num_q_heads;
  a.hkv = cfg->num_kv_heads;
  a.g = cfg->num_q_heads / cfg->num_kv_heads;
  a.tail_k = static_cast<const __half*>(tail_k);
  a.tail_v = static_cast<const __half*>(tail_v);
  a.scale = softmax_scale;
  a.out = static_cast<__half*>(out);
  a.ws_part = p.nsplit > 1 ? static_cast<float*>(workspace) : nullptr;
  a.ws_count = p.nsplit > 1
                   ? reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + p.part_bytes)
                   : nullptr;
  a.pages_per_split = p.pages_per_split;
  a.nsplit = p.nsplit;
  a.cluster = p.cluster ? 1 : 0;
  a.fmt = cfg_fmt(cfg);
  a.status = status;
  cudaError_t e = decode_mma_supported(a.g) ? launch_decode_mma(a, (cudaStream_t)stream)
                                            : launch_decode_simple(a, (cudaStream_t)stream);
  return e == cudaSuccess ? KVARN_OK : KVARN_ERR_LAUNCH;
}

int kvarn_chunk_attention(const kvarn_config_t* cfg, const void* q, int chunk_max,
                          const int32_t* start, const int32_t* chunk_lens, int batch,
                          int max_seq, const void* pool, int64_t num_pages,
                          const int32_t* block_table, int max_blocks, const void* tail_k,
                          const void* tail_v, float softmax_scale, void* out, int32_t* status,
                          kvarn_stream_t stream) {
  int rc = kvarn_config_validate(cfg);
  if (rc != KVARN_OK) return rc;
  if (batch < 0 || chunk_max < 0 || max_seq < 0 || max_blocks < 0 || num_pages < 0)
    return KVARN_ERR_INVALID_ARG;
  if (batch == 0 || chunk_max == 0) return KVARN_OK;
  if (!q || !start || !chunk_lens || !tail_k || !tail_v || !out) return KVARN_ERR_INVALID_ARG;
  if (max_seq >= kT && (!pool || !block_table || num_pages <= 0 || max_blocks < max_seq / kT))
    return KVARN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(pool) || !aligned16(tail_k) || !aligned16(tail_v) ||
      !aligned16(out))
    return KVARN_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || softmax_scale != softmax_scale) return KVARN_ERR_INVALID_ARG;
  const int g = cfg->num_q_heads / cfg->num_kv_heads;
  const int tq = chunk_rows_per_tile(g);
  const int64_t ntq = ((int64_t)chunk_max + tq - 1) / tq;
  if (batch > 65535 || cfg->num_kv_heads > 65535 || ntq > 0x7fffffff) return KVARN_ERR_UNSUPPORTED;
  ChunkArgs a;
  a.q = static_cast<const __half*>(q);
  a.M = chunk_max;
  a.start = start;
  a.chunk_lens = chunk_lens;
  a.batch = batch;
  a.max_seq = max_seq;
  a.hq = cfg->num_q_heads;
  a.hkv = cfg->num_kv_heads;
  a.g = g;
  a.tq = tq;
  a.ntq = (int)ntq;
  a.pool = static_cast<const uint8_t*>(pool);
  a.num_pages = num_pages;
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.tail_k = static_cast<const __half*>(tail_k);
  a.tail_v = static_cast<const __half*>(tail_v);
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.out = static_cast<__half*>(out);
  a.fmt = cfg_fmt(cfg);
  a.status = status;
  return launch_chunk_attention(a, (cudaStream_t)stream) == cudaSuccess ? KVARN_OK
                                                                         : KVARN_ERR_LAUNCH;
}

int kvarn_fp16_write_blocks(const void* k, const void* v, int64_t stride_b, int64_t stride_t,
                            int64_t stride_h, int batch, int num_kv_heads,
                            const int32_t* seq_lens, int max_seq, const int32_t* block_table,
                            int max_blocks, void* pool, int64_t num_pages, int32_t* status,
                            kvarn_stream_t stream) {
  if (batch < 0 || max_seq < 0 || max_blocks < 0 || num_pages < 0 || num_kv_heads <= 0)
    return KVARN_ERR_INVALID_ARG;
  if (batch == 0 || max_seq == 0) return KVARN_OK;
  if (!k || !v || !seq_lens || !block_table || !pool || num_pages <= 0)
    return KVARN_ERR_INVALID_ARG;
  if ((int64_t)max_blocks * kT < (int64_t)max_seq) return KVARN_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(pool)) return KVARN_ERR_INVALID_ARG;
  if (stride_b < 0 || stride_t < kD || stride_h < kD || (stride_b | stride_t | stride_h) % 8)
    return KVARN_ERR_INVALID_ARG;
  if (num_kv_heads > 65535 || batch > 65535) return KVARN_ERR_UNSUPPORTED;
  F16WriteArgs a;
  a.k = static_cast<const __half*>(k);
  a.v = static_cast<const __half*>(v);
  a.sb = stride_b;
  a.st = stride_t;
  a.sh = stride_h;
  a.batch = batch;
  a.hkv = num_kv_heads;
  a.max_seq = max_seq;
  a.seq_lens = seq_lens;
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.pool = static_cast<uint8_t*>(pool);
  a.num_pages = num_pages;
  a.status = status;
  return launch_fp16_write(a, (cudaStream_t)stream) == cudaSuccess ? KVARN_OK : KVARN_ERR_LAUNCH;
}

size_t kvarn_fp16_decode_workspace_bytes(int num_q_heads, int num_kv_heads, int batch,
                                         int max_seq) {
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads || batch <= 0 ||
      max_seq < 0)
    return 0;
  const int sms = device_sm_count();
  if (sms <= 0) return 0;
  const DecodePlan p = fp16_decode_plan(batch, num_q_heads, num_kv_heads, max_seq, sms);
  return p.part_bytes + p.count_bytes;
}

int kvarn_fp16_decode_attention(const void* q, int num_q_heads, int num_kv_heads,
                                const void* pool, int64_t num_pages, const int32_t* block_table,
                                int max_blocks, const int32_t* seq_lens, int batch, int max_seq,
                                float softmax_scale, void* out, void* workspace,
                                size_t workspace_bytes, int32_t* status, kvarn_stream_t stream) {
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads)
    return KVARN_ERR_INVALID_ARG;
  if (num_q_heads / num_kv_heads > 8) return KVARN_ERR_UNSUPPORTED;
  if (batch < 0 || max_seq < 0 || max_blocks < 0 || num_pages < 0) return KVARN_ERR_INVALID_ARG;
  if (batch == 0) return KVARN_OK;
  if (!q || !seq_lens || !out) return KVARN_ERR_INVALID_ARG;
  if (max_seq > 0 && (!pool || !block_table || num_pages <= 0 ||
                      (int64_t)max_blocks * kT < (int64_t)max_seq))
    return KVARN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(pool) || !aligned16(out) || !aligned16(workspace))
    return KVARN_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || softmax_scale != softmax_scale) return KVARN_ERR_INVALID_ARG;
  if (batch > 65535 || num_kv_heads > 65535 || num_pages > 0x7fffffff)
    return KVARN_ERR_UNSUPPORTED;
  const int sms = device_sm_count();
  if (sms <= 0) return KVARN_ERR_LAUNCH;
  const DecodePlan p = fp16_decode_plan(batch, num_q_heads, num_kv_heads, max_seq, sms);
  if (p.nsplit > 1 && (!workspace || workspace_bytes < p.part_bytes + p.count_bytes))
    return KVARN_ERR_WORKSPACE;
  F16DecodeArgs a;
  a.q = static_cast<const __half*>(q);
  a.num_pages = num_pages;
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.seq_lens = seq_lens;
  a.batch = batch;
  a.max_seq = max_seq;
  a.hq = num_q_heads;
  a.hkv = num_kv_heads;
  a.g = num_q_heads / num_kv_heads;
  a.scale = softmax_scale;
  a.out = static_cast<__half*>(out);
  a.ws_part = p.nsplit > 1 ? static_cast<float*>(workspace) : nullptr;
  a.ws_count = p.nsplit > 1
                   ? reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + p.part_bytes)
                   : nullptr;
  a.pages_per_split = p.pages_per_split;
  a.nsplit = p.nsplit;
  a.status = status;
  return launch_fp16_decode(a, pool, (cudaStream_t)stream) == cudaSuccess ? KVARN_OK
                                                                          : KVARN_ERR_LAUNCH;
}

int kvarn_fp8_write_blocks(const void* k, const void* v, int64_t stride_b, int64_t stride_t,
                            int64_t stride_h, int batch, int num_kv_heads,
                            const int32_t* seq_lens, int max_seq, const int32_t* block_table,
                            int max_blocks, void* pool, int64_t num_pages, int32_t* status,
                            kvarn_stream_t stream) {
  if (batch < 0 || max_seq < 0 || max_blocks < 0 || num_pages < 0 || num_kv_heads <= 0)
    return KVARN_ERR_INVALID_ARG;
  if (batch == 0 || max_seq == 0) return KVARN_OK;
  if (!k || !v || !seq_lens || !block_table || !pool || num_pages <= 0)
    return KVARN_ERR_INVALID_ARG;
  if ((int64_t)max_blocks * kT < (int64_t)max_seq) return KVARN_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(pool)) return KVARN_ERR_INVALID_ARG;
  if (stride_b < 0 || stride_t < kD || stride_h < kD || (stride_b | stride_t | stride_h) % 8)
    return KVARN_ERR_INVALID_ARG;
  if (num_kv_heads > 65535 || batch > 65535) return KVARN_ERR_UNSUPPORTED;
  F16WriteArgs a;
  a.k = static_cast<const __half*>(k);
  a.v = static_cast<const __half*>(v);
  a.sb = stride_b;
  a.st = stride_t;
  a.sh = stride_h;
  a.batch = batch;
  a.hkv = num_kv_heads;
  a.max_seq = max_seq;
  a.seq_lens = seq_lens;
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.pool = static_cast<uint8_t*>(pool);
  a.num_pages = num_pages;
  a.status = status;
  return launch_fp8_write(a, (cudaStream_t)stream) == cudaSuccess ? KVARN_OK : KVARN_ERR_LAUNCH;
}

size_t kvarn_fp8_decode_workspace_bytes(int num_q_heads, int num_kv_heads, int batch,
                                         int max_seq) {
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads || batch <= 0 ||
      max_seq < 0)
    return 0;
  const int sms = device_sm_count();
  if (sms <= 0) return 0;
  const DecodePlan p = fp8_decode_plan(batch, num_q_heads, num_kv_heads, max_seq, sms);
  return p.part_bytes + p.count_bytes;
}

int kvarn_fp8_decode_attention(const void* q, int num_q_heads, int num_kv_heads,
                                const void* pool, int64_t num_pages, const int32_t* block_table,
                                int max_blocks, const int32_t* seq_lens, int batch, int max_seq,
                                float softmax_scale, void* out, void* workspace,
                                size_t workspace_bytes, int32_t* status, kvarn_stream_t stream) {
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads)
    return KVARN_ERR_INVALID_ARG;
  if (num_q_heads / num_kv_heads > 8) return KVARN_ERR_UNSUPPORTED;
  if (batch < 0 || max_seq < 0 || max_blocks < 0 || num_pages < 0) return KVARN_ERR_INVALID_ARG;
  if (batch == 0) return KVARN_OK;
  if (!q || !seq_lens || !out) return KVARN_ERR_INVALID_ARG;
  if (max_seq > 0 && (!pool || !block_table || num_pages <= 0 ||
                      (int64_t)max_blocks * kT < (int64_t)max_seq))
    return KVARN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(pool) || !aligned16(out) || !aligned16(workspace))
    return KVARN_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || softmax_scale != softmax_scale) return KVARN_ERR_INVALID_ARG;
  if (batch > 65535 || num_kv_heads > 65535 || num_pages > 0x7fffffff)
    return KVARN_ERR_UNSUPPORTED;
  const int sms = device_sm_count();
  if (sms <= 0) return KVARN_ERR_LAUNCH;
  const DecodePlan p = fp8_decode_plan(batch, num_q_heads, num_kv_heads, max_seq, sms);
  if (p.nsplit > 1 && (!workspace || workspace_bytes < p.part_bytes + p.count_bytes))
    return KVARN_ERR_WORKSPACE;
  F16DecodeArgs a;
  a.q = static_cast<const __half*>(q);
  a.num_pages = num_pages;
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.seq_lens = seq_lens;
  a.batch = batch;
  a.max_seq = max_seq;
  a.hq = num_q_heads;
  a.hkv = num_kv_heads;
  a.g = num_q_heads / num_kv_heads;
  a.scale = softmax_scale;
  a.out = static_cast<__half*>(out);
  a.ws_part = p.nsplit > 1 ? static_cast<float*>(workspace) : nullptr;
  a.ws_count = p.nsplit > 1
                   ? reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + p.part_bytes)
                   : nullptr;
  a.pages_per_split = p.pages_per_split;
  a.nsplit = p.nsplit;
  a.status = status;
  return launch_fp8_decode(a, pool, (cudaStream_t)stream) == cudaSuccess ? KVARN_OK
                                                                          : KVARN_ERR_LAUNCH;
}

size_t kvarn_snapkv_workspace_bytes(const kvarn_config_t* cfg, int batch, int window,
                                     int max_seq) {
  if (kvarn_config_validate(cfg) != KVARN_OK || batch <= 0 || window <= 0 || max_seq <= 0)
    return 0;
  const int g = cfg->num_q_heads / cfg->num_kv_heads;
  const int64_t nrt = ((int64_t)window * g + 127) / 128;
  const int64_t nchunks = ((int64_t)max_seq + kSnapChunkTiles * 128 - 1) / (kSnapChunkTiles * 128);
  const size_t stats = ((size_t)batch * cfg->num_kv_heads * nrt * nchunks * 256 * 4 + 255) & ~(size_t)255;
  const size_t pooled = ((size_t)batch * cfg->num_kv_heads * max_seq * 4 + 255) & ~(size_t)255;
  return stats + pooled;
}

int kvarn_snapkv_select(const kvarn_config_t* cfg, const void* q_window, int window,
                        const void* k, int64_t stride_b, int64_t stride_t, int64_t stride_h,
                        const int32_t* seq_lens, int batch, int max_seq, int capacity,
                        int pool_kernel, float softmax_scale, float* votes, int32_t* indices,
                        void* workspace, size_t workspace_bytes, int32_t* status,
                        kvarn_stream_t stream) {
  int rc = kvarn_config_validate(cfg);
  if (rc != KVARN_OK) return rc;
  if (batch < 0 || max_seq < 0 || window <= 0 || capacity < window || pool_kernel < 1 ||
      pool_kernel % 2 == 0)
    return KVARN_ERR_INVALID_ARG;
  if (batch == 0 || max_seq == 0) return KVARN_OK;
  if (!q_window || !k || !seq_lens || !votes || !indices || !workspace)
    return KVARN_ERR_INVALID_ARG;
  if (!aligned16(q_window) || !aligned16(k) || !aligned16(workspace) ||
      ((uintptr_t)votes & 3) || ((uintptr_t)indices & 3))
    return KVARN_ERR_INVALID_ARG;
  if (stride_b < 0 || stride_t < kD || stride_h < kD || (stride_b | stride_t | stride_h) % 8)
    return KVARN_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || softmax_scale != softmax_scale) return KVARN_ERR_INVALID_ARG;
  if (batch > 65535 || cfg->num_kv_heads > 65535) return KVARN_ERR_UNSUPPORTED;
  const size_t need = kvarn_snapkv_workspace_bytes(cfg, batch, window, max_seq);
  if (workspace_bytes < need) return KVARN_ERR_WORKSPACE;
  SnapArgs a;
  a.q = static_cast<const __half*>(q_window);
  a.W = window;
  a.batch = batch;
  a.max_seq = max_seq;
  a.hq = cfg->num_q_heads;
  a.hkv = cfg->num_kv_heads;
  a.g = cfg->num_q_heads / cfg->num_kv_heads;
  a.seq_lens = seq_lens;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.nrt = (window * a.g + 127) / 128;
  a.nchunks = (max_seq + kSnapChunkTiles * 128 - 1) / (kSnapChunkTiles * 128);
  a.stats = static_cast<float*>(workspace);
  const size_t stats = ((size_t)batch * a.hkv * a.nrt * a.nchunks * 256 * 4 + 255) & ~(size_t)255;
  a.votes = votes;
  a.status = status;
  CUtensorMap tm;
  if (!encode_kv_tile_map(&tm, k, stride_b, stride_t, stride_h, batch, max_seq, a.hkv, &a.roles))
    return KVARN_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  if (launch_snapkv_scores(a, tm, 0, s) != cudaSuccess) return KVARN_ERR_LAUNCH;
  if (launch_snapkv_scores(a, tm, 1, s) != cudaSuccess) return KVARN_ERR_LAUNCH;
  SnapSelectArgs sa;
  sa.votes = votes;
  sa.pooled = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + stats);
  sa.seq_lens = seq_lens;
  sa.batch = batch;
  sa.hkv = a.hkv;
  sa.max_seq = max_seq;
  sa.W = window;
  sa.capacity = capacity;
  sa.kernel = pool_kernel;
  sa.indices = indices;
  return launch_snapkv_select(sa, s) == cudaSuccess ? KVARN_OK : KVARN_ERR_LAUNCH;
}

int kvarn_snapkv_gather(const void* k, const void* v, int64_t stride_b, int64_t stride_t,
                        int64_t stride_h, int batch, int max_seq, int num_kv_heads,
                        const int32_t* indices, int capacity, void* k_out, void* v_out,
                        kvarn_stream_t stream) {
  if (batch < 0 || max_seq < 0 || num_kv_heads <= 0 || capacity < 0)
    return KVARN_ERR_INVALID_ARG;
  if (batch == 0 || capacity == 0) return KVARN_OK;
  if (!k || !v || !indices || !k_out || !v_out) return KVARN_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_out) || !aligned16(v_out))
    return KVARN_ERR_INVALID_ARG;
  if (stride_b < 0 || stride_t < kD || stride_h < kD || (stride_b | stride_t | stride_h) % 8)
    return KVARN_ERR_INVALID_ARG;
  if (batch > 65535 || num_kv_heads > 65535) return KVARN_ERR_UNSUPPORTED;
  return launch_snapkv_gather(static_cast<const __half*>(k), static_cast<const __half*>(v),
                              stride_b, stride_t, stride_h, batch, max_seq, num_kv_heads,
                              indices, capacity, static_cast<__half*>(k_out), static_cast<__half*>(v_out),
                              (cudaStream_t)stream) == cudaSuccess
             ? KVARN_OK
             : KVARN_ERR_LAUNCH;
}

int kvarn_dequantize_pages(const void* records, int64_t n, float* yk, float* yv,
                           kvarn_stream_t stream) {
  if (n < 0) return KVARN_ERR_INVALID_ARG;
  if (n == 0) return KVARN_OK;
  if (!records || !yk || !yv || !aligned16(records) || n > 0x7fffffff)
    return KVARN_ERR_INVALID_ARG;
  return launch_dequantize(kFmtF32, static_cast<const uint8_t*>(records), n, yk, yv,
                           (cudaStream_t)stream) == cudaSuccess
             ? KVARN_OK
             : KVARN_ERR_LAUNCH;
}

int kvarn_wait_check(int32_t* status, int arrive, uint32_t limit_us, kvarn_stream_t stream) {
  if (!status || (arrive != 0 && arrive != 1) || limit_us == 0 || limit_us > 1000000u)
    return KVARN_ERR_INVALID_ARG;
  return launch_wait_check(status, (uint64_t)limit_us * 1000u, arrive, (cudaStream_t)stream) ==
                 cudaSuccess
             ? KVARN_OK
             : KVARN_ERR_LAUNCH;
}

int kvarn_dequantize_records(const kvarn_config_t* cfg, const void* records, int64_t n,
                             float* yk, float* yv, kvarn_stream_t stream) {
  const int rc = kvarn_config_validate(cfg);
  if (rc != KVARN_OK) return rc;
  if (n < 0) return KVARN_ERR_INVALID_ARG;
  if (n == 0) return KVARN_OK;
  if (!records || !yk || !yv || !aligned16(records) || n > 0x7fffffff)
    return KVARN_ERR_INVALID_ARG;
  return launch_dequantize(cfg_fmt(cfg), static_cast<const uint8_t*>(records), n, yk, yv,
                           (cudaStream_t)stream) == cudaSuccess
             ? KVARN_OK
             : KVARN_ERR_LAUNCH;
}

const char* kvarn_status_string(int code) {
  switch (code) {
    case KVARN_OK: return "ok";
    case KVARN_ERR_INVALID_ARG: return "invalid argument";
    case KVARN_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVARN_ERR_WORKSPACE: return "decode workspace missing or too small";
    case KVARN_ERR_LAUNCH: return "CUDA launch failed";
    case KVARN_STATUS_BAD_PAGE: return "device: block-table entry outside the pool";
    case KVARN_STATUS_BAD_LENGTH: return "device: sequence length beyond max_seq or the table";
    case KVARN_STATUS_TIMEOUT: return "device: a bounded wait gave up";
    default: return code > 0 ? "device: several status bits set" : "unknown error";
  }
}

const char* kvarn_version(void) { return "0.1.0"; }

}  // extern "C"
