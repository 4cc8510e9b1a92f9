/*
 * kvarn.h -- C ABI of the KVarN-style quantized KV cache for B300 (sm_103a).
 *
 * What it computes.  "KVarN: Huawei'den KV-Cache Kuantizasyonu icin Yerel vLLM
 * Backend'i" (blog.edumints.com), section "KVarN Nasil Calisir?" (How KVarN
 * works): the KV cache is quantized in fixed-size token blocks, and each block
 * goes through an orthonormal Hadamard rotation along channels, a Sinkhorn-like
 * row/column variance normalization in the log domain, and asymmetric
 * round-to-nearest with 4-bit keys and 2-bit values (format kvarn_k4v2_g128,
 * section "Yazilim Gelistirme ve Ogrenme Acisindan Pratik Cikarimlar").  The
 * quantized blocks live in a paged pool addressed through a block table, as in
 * "KV Cache (Anahtar-Deger Onbellegi)" (yapayzekasozluk.tr), section "Paged
 * Attention (vLLM)"; decode attention reads every cached token of a sequence
 * for one new query token ("KV Cache Nasil Calisir?"), several query heads
 * sharing one KV head (GQA, "Sik Sorulan Sorular").
 *
 * Fixed readings (the pages leave these open):
 *   head_dim = block = group = 128; one block = 128 tokens x 128 channels of one
 *   KV head; K and V are separate tiles.  H = Sylvester Hadamard / sqrt(128),
 *   y_t = H x_t.  Sinkhorn: rows = tokens, columns = channels, K iterations of
 *   (row step, column step), each step sets the log scale so that the centred
 *   population std of Y * exp(-a_t - b_d) becomes 1 along that axis, skipping a
 *   row/column whose variance is <= 1e-10 * its mean square.  Groups are the 128
 *   channels of one token: z = min, s = (max - min) / (2^bits - 1),
 *   q = rint((x - z) / s) (ties to even).  Metadata fp32, row scale folded in:
 *   dequantized rotated value yhat_td = c_d * (s'_t * q_td + z'_t).
 *
 * Page record: one per (page, KV head), KVARN_PAGE_BYTES bytes, 16-byte aligned;
 * the K part then the V part, each contiguous (codes, row metadata, column
 * scales), so that a reader can fetch either part with one bulk copy:
 *   [0,     8192) K codes, token-major: token t at 64 t; byte j = channel 2j
 *                 (bits 0-3) | channel 2j+1 (bits 4-7)
 *   [8192,  9216) K {s', z'} fp32 per token (token t at 8192 + 8 t)
 *   [9216,  9728) K column scale c_d fp32
 *   [9728, 13824) V codes, 2 bits each, 1024 little-endian 32-bit words:
 *                 with channel c = 16m + 8e + r (m < 8, e < 2, r < 8) and
 *                 token t = 16k + 8f + 2j + s (k < 8, f < 2, j < 4, s < 2),
 *                 the code of (c, t) is bits 2i, 2i+1 with i = 2(k mod 4) +
 *                 f + 8s of word 128m + 16r + 4j + 2e + floor(k/4) (a fixed
 *                 permutation of channel-major order that lets a decode warp
 *                 fetch each tensor-core fragment with one 16-byte load)
 *   [13824,14848) V {s', z'} fp32 per token
 *   [14848,15360) V column scale c_d fp32
 * Format variant "_m16" (config meta_fp16 = 1; 108 bytes per token-head
 * instead of 120): the same codes and the same fp32 arithmetic, with every
 * stored s', z', c_d rounded once more to fp16 (round to nearest even; a
 * value beyond fp16's range becomes infinity, so inputs whose scales exceed
 * it need the fp32 format).  Record of KVARN_PAGE_BYTES_M16 bytes:
 *   [0,     8192) K codes (as above)
 *   [8192,  8704) K {s', z'} fp16 per token (token t at 8192 + 4 t)
 *   [8704,  8960) K column scale c_d fp16
 *   [8960, 13056) V codes (the same permutation)
 *   [13056,13568) V {s', z'} fp16 per token
 *   [13568,13824) V column scale c_d fp16
 * Format variant "_pc" (config per_channel = 1; fp32 metadata, 15360 bytes):
 * after the same rotation and normalization, one RTN group is one channel's
 * 128 tokens of the tile, so the row scale r_t is stored per token and c_d
 * folds into the per-channel scale and zero: with x_td = Y_td / (r_t c_d),
 * z_d = min_t x_td, s_d = (max_t - min_t) / (2^bits - 1), and
 * yhat_td = r_t * (cs_d * q_td + cz_d), cs_d = c_d s_d, cz_d = c_d z_d:
 *   [0,     8192) K codes (as above)
 *   [8192,  8704) K r_t fp32 per token
 *   [8704,  9728) K {cs_d, cz_d} fp32 per channel
 *   [9728, 13824) V codes (the same permutation)
 *   [13824,14336) V r_t fp32 per token
 *   [14336,15360) V {cs_d, cz_d} fp32 per channel
 * Format variant "k4v2_g64" (config group = 64; fp32 metadata, 17408 bytes,
 * 136 B per token-head): the same stages with two RTN groups per token,
 * channels 0-63 and 64-127, each with its own {s', z'} (row scale folded in):
 *   [0,     8192) K codes (as above)
 *   [8192, 10240) K {s'_0, z'_0, s'_1, z'_1} fp32 per token (token t at 8192 + 16 t)
 *   [10240,10752) K column scale c_d fp32
 *   [10752,14848) V codes (the same permutation)
 *   [14848,16896) V {s'_0, z'_0, s'_1, z'_1} fp32 per token
 *   [16896,17408) V column scale c_d fp32
 * Format variant "k4v4_g128" (config v_bits = 4; fp32 metadata, 19456 bytes,
 * 152 B per token-head): the same stages with 4-bit RTN on V as on K.  The K
 * part is as above; the V part holds 4-bit codes in their own permutation:
 * with channel c = 16m + 8e + r and token t = 16k + 8f + 2j + s, the code of
 * (c, t) is nibble 4s + 2(k mod 2) + f (bits 4n of a little-endian word) of
 * word 256m + 32r + 8j + 4e + floor(k/2):
 *   [9728, 17920) V codes, 2048 32-bit words
 *   [17920,18944) V {s', z'} fp32 per token
 *   [18944,19456) V column scale c_d fp32
 * Format variant "k8v4_g128" (config k_bits = 8, v_bits = 4; fp32 metadata,
 * 27648 bytes, 216 B per token-head): 8-bit RTN on K (2^8 - 1 steps), V as in
 * "k4v4_g128".  K codes are one byte per channel, token-major rows of 128
 * bytes whose 16-byte chunks trade places pairwise in odd tokens: channel d
 * of token t is byte 128 t + (d XOR 16 (t mod 2)):
 *   [0,    16384) K codes
 *   [16384,17408) K {s', z'} fp32 per token
 *   [17408,17920) K column scale c_d fp32
 *   [17920,26112) V codes (the 4-bit permutation above)
 *   [26112,27136) V {s', z'} fp32 per token
 *   [27136,27648) V column scale c_d fp32
 * Pool = [num_pages][num_kv_heads][kvarn_page_bytes(cfg)].  The newest len mod 128
 * tokens of a sequence stay fp16 in a caller-owned tail buffer
 * [B][num_kv_heads][128 slots][128] per K and V.
 *
 * Conventions for every call:
 *   - the library allocates nothing and keeps no state between calls that
 *     affects a result (it remembers, per device, launch settings it has
 *     already applied; kvarn_decode_attention_noalloc's scratch is a fixed
 *     array, see there); calls are safe from several host threads; every
 *     pointer is caller-owned DEVICE memory unless stated otherwise;
 *   - every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and never synchronises;
 *   - the return value is KVARN_OK or a negative KVARN_ERR_*; all argument
 *     checks run on the host before any launch, and a failed check launches
 *     nothing;
 *   - errors found on the device (a page id outside [0, num_pages), a length
 *     beyond the table, a wait that gave up) are OR-ed into `*status`
 *     (nullable, device int32, caller zeroes it) as KVARN_STATUS_* bits; the
 *     offending unit is skipped, nothing traps;
 *   - fp16 means IEEE binary16; all tensors are little-endian and densely
 *     packed in their last dimension.
 */
#ifndef KVARN_H
#define KVARN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *kvarn_stream_t; /* identical to cudaStream_t */

#define KVARN_HEAD_DIM 128
#define KVARN_BLOCK_TOKENS 128
#define KVARN_PAGE_BYTES 15360
#define KVARN_PAGE_BYTES_M16 13824
#define KVARN_PAGE_BYTES_G64 17408
#define KVARN_PAGE_BYTES_V4 19456
#define KVARN_PAGE_BYTES_K8 27648

/* return codes */
#define KVARN_OK 0
#define KVARN_ERR_INVALID_ARG (-1) /* null/misaligned pointer, bad size or stride */
#define KVARN_ERR_UNSUPPORTED (-2) /* a format or shape this library does not run */
#define KVARN_ERR_WORKSPACE (-3)   /* decode workspace missing or too small */
#define KVARN_ERR_LAUNCH (-4)      /* the CUDA launch itself failed */

/* device status bits, OR-ed into *status */
#define KVARN_STATUS_BAD_PAGE 1    /* block-table entry outside [0, num_pages) */
#define KVARN_STATUS_BAD_LENGTH 2  /* sequence length beyond max_seq or the table */
#define KVARN_STATUS_TIMEOUT 4     /* a bounded wait on the device gave up */

typedef struct {
    int head_dim;       /* 128 */
    int block_tokens;   /* 128 */
    int group;          /* 128: quantization group = one token's channels; 64:
                           format variant "k4v2_g64", two groups per token
                           (fp32 metadata, not with "_pc") */
    int k_bits;         /* 4; 8: format variant "k8v4_g128" (with v_bits = 4,
                           fp32 metadata, groups of 128) */
    int v_bits;         /* 2; 4: format variant "k4v4_g128" (fp32 metadata,
                           groups of 128, not with "_pc") */
    int sinkhorn_iters; /* 0..64; 2 from the iteration-selection rule */
    int num_q_heads;    /* Hq, a multiple of num_kv_heads */
    int num_kv_heads;   /* Hkv; Hq / Hkv <= 16 */
    int sinkhorn_rms;   /* 0: centred std (default); 1: format variant "_rms",
                           the uncentred root mean square (Sinkhorn-Knopp on
                           the squares; only all-zero rows/columns skipped).
                           The page record is the same either way. */
    int meta_fp16;      /* 0: fp32 metadata (default); 1: format variant "_m16",
                           metadata stored as fp16 (KVARN_PAGE_BYTES_M16) */
    int per_channel;    /* 0: per-token RTN groups (default); 1: format variant
                           "_pc", per-channel groups (fp32 metadata only) */
} kvarn_config_t;

/* Fills *out from a format string: "k4v2_g128" or "kvarn_k4v2_g128" (the
 * KVarN page's --kv-cache-dtype value), or "k4v2_g64" / "kvarn_k4v2_g64" for
 * groups of 64 channels, or "k4v4_g128" for 4-bit values, or "k8v4_g128"
 * for 8-bit keys and 4-bit values, optionally followed by the variant
 * suffixes "_rms" (the uncentred statistic), "_m16" (fp16 metadata) and "_pc"
 * (per-channel groups; not with "_m16"), each at most once and in any order,
 * and then "_s<K>" to set the Sinkhorn iteration count.  Returns KVARN_ERR_UNSUPPORTED for any other format,
 * KVARN_ERR_INVALID_ARG for bad head counts or a null pointer. */
int kvarn_config_from_string(const char *s, int num_q_heads, int num_kv_heads,
                             kvarn_config_t *out);

/* KVARN_OK if the configuration is one this library runs. */
int kvarn_config_validate(const kvarn_config_t *cfg);

/* Bytes of one page record (per page and KV head): KVARN_PAGE_BYTES (15360),
 * KVARN_PAGE_BYTES_M16 (13824) for the "_m16" format, KVARN_PAGE_BYTES_G64
 * (17408) for groups of 64, KVARN_PAGE_BYTES_V4 (19456) for 4-bit values, or
 * KVARN_PAGE_BYTES_K8 (27648) for 8-bit keys with 4-bit values; 0 on a bad
 * config.
 * Every call that takes a pool reads it with this record size. */
size_t kvarn_page_bytes(const kvarn_config_t *cfg);

/* Prefill quantization ("KVarN Nasil Calisir?", all four stages).
 *   k, v        fp16 [B][S][Hkv][128], element (b,t,h,c) at
 *               b*stride_b + t*stride_t + h*stride_h + c; 16-byte aligned,
 *               strides multiples of 8 elements
 *   seq_lens    int32 [batch], tokens of each sequence (<= max_seq); k and v
 *               must hold that many tokens (the library cannot see their size)
 *   max_seq     host upper bound on seq_lens, sizes the grid
 *   block_table int32 [batch][max_blocks]; block j of sequence b goes to page
 *               block_table[b*max_blocks + j]; needs max_blocks >= max_seq/128
 *   pool        [num_pages][Hkv][15360] bytes, written for every full block
 *   tail_k/_v   fp16 [batch][Hkv][128][128]: the len mod 128 leftover tokens
 *               of each sequence are copied to slots 0..len%128-1
 * Every full block of 128 tokens is quantized: K to 4 bits, V to 2 bits. */
int kvarn_quantize_blocks(const kvarn_config_t *cfg, const void *k, const void *v,
                          int64_t stride_b, int64_t stride_t, int64_t stride_h, int batch,
                          const int32_t *seq_lens, int max_seq, const int32_t *block_table,
                          int max_blocks, void *pool, int64_t num_pages, void *tail_k,
                          void *tail_v, int32_t *status, kvarn_stream_t stream);

/* Decode-time append of one token per sequence ("KV Cache Nasil Calisir?":
 * only the new token's K,V are computed and added to the cache).
 *   k_new, v_new fp16 [batch][Hkv][128]
 *   pos          int32 [batch]: the sequence length before this append; the
 *                token goes to tail slot pos % 128; pos < 0 skips the sequence
 *   When the slot is 127 the full tail is quantized (all four stages) into page
 *   block_table[b*max_blocks + pos/128] in the same launch, so the page must
 *   already be in the table.  The caller advances pos / seq_lens afterwards. */
int kvarn_append_token(const kvarn_config_t *cfg, const void *k_new, const void *v_new,
                       const int32_t *pos, int batch, const int32_t *block_table,
                       int max_blocks, void *pool, int64_t num_pages, void *tail_k,
                       void *tail_v, int32_t *status, kvarn_stream_t stream);

/* The split-K plan decode uses for (batch, max_seq) on a GPU with `num_sms`
 * streaming multiprocessors (num_sms <= 0: the current device's count).  The
 * pages of each (sequence, KV head) are cut into *nsplit runs of
 * *pages_per_split pages, as many as keep the whole grid resident at once.
 * When the (sequence, KV head) pairs alone outnumber the CTAs that can be
 * resident at once (at most 8 query heads per KV head), the grid runs in
 * several waves and runs are cut to at most 32 pages instead, as far as the
 * partial states fit KVARN_NOALLOC_SCRATCH_BYTES, so that long sequences of
 * a ragged batch do not straggle.  *workspace_bytes is the decode workspace that plan needs
 * (0: none).  Any output pointer may be NULL.  Host arithmetic only when
 * num_sms > 0 (no CUDA call); KVARN_ERR_LAUNCH when num_sms <= 0 and no
 * device answers. */
int kvarn_decode_split_plan(const kvarn_config_t *cfg, int batch, int max_seq, int num_sms,
                            int *pages_per_split, int *nsplit, size_t *workspace_bytes);

/* Bytes of decode workspace for (batch, max_seq) on the current device: the
 * plan above for that device's SM count.  0 when no split is needed, and 0
 * when no CUDA device is current (nothing can launch then either). */
size_t kvarn_decode_workspace_bytes(const kvarn_config_t *cfg, int batch, int max_seq);

/* Decode attention for one new query token per sequence:
 *   out[b][h] = sum_t softmax_t(scale * q[b][h] . k_t) v_t
 * over the len/128 quantized pages of sequence b (keys and values dequantized
 * and rotated back: attention scores are unchanged by the orthonormal
 * rotation, KVarN page stage 2) followed by its len%128 fp16 tail tokens.
 * Query head h reads KV head h / (Hq/Hkv).
 *   q          fp16 [batch][Hq][128]
 *   seq_lens   int32 [batch], total tokens (pages + tail), <= max_seq
 *   out        fp16 [batch][Hq][128]; a sequence of length 0 gives zeros
 *   workspace  >= kvarn_decode_workspace_bytes(cfg, batch, max_seq) bytes,
 *              16-byte aligned, ZERO-FILLED before its first use; every call
 *              leaves it zero-filled again in its counter region, so one
 *              buffer serves any number of calls on one stream (calls that
 *              share a workspace must not overlap on the GPU).
 * The work is split across CTAs along each sequence's pages (split-K) and the
 * partial softmax states are merged with a log-sum-exp in the same launch:
 * inside a thread-block cluster (distributed shared memory) when a sequence
 * has 2 to 4 splits in a grid of one wave, through the workspace
 * otherwise.  The launch then uses thread-block clusters, so the GPU must be
 * able to co-schedule up to 4 CTAs of the kernel; a launch failure returns
 * KVARN_ERR_LAUNCH. */
int kvarn_decode_attention(const kvarn_config_t *cfg, const void *q, const void *pool,
                           int64_t num_pages, const int32_t *block_table, int max_blocks,
                           const int32_t *seq_lens, int batch, int max_seq,
                           const void *tail_k, const void *tail_v, float softmax_scale,
                           void *out, void *workspace, size_t workspace_bytes,
                           int32_t *status, kvarn_stream_t stream);

/* Size of the scratch array built into the library for
 * kvarn_decode_attention_noalloc: 16 MiB, held on every GPU that loads it.
 * On a 148-SM B300 every configuration with Hq/Hkv <= 16 fits in it whatever
 * its batch and lengths (a plan of one wave needs at most 3.8 MB, and a plan
 * of several waves is sized to it); a GPU with many more SMs may plan more. */
#define KVARN_NOALLOC_SCRATCH_BYTES (16u << 20)

/* Decode attention without any caller-provided workspace.  The pages have no
 * counterpart to this call; it exists for callers that cannot allocate GPU
 * memory, such as plugin hosts that hand a kernel only its inputs and outputs,
 * or serving loops that cannot afford the device synchronisation cudaMalloc
 * brings.  It computes exactly what kvarn_decode_attention computes, with the
 * same arguments minus the workspace, using instead a fixed array of
 * KVARN_NOALLOC_SCRATCH_BYTES inside the library.
 *   - Returns KVARN_ERR_WORKSPACE, launching nothing, when (batch, max_seq)
 *     would need more scratch than that (kvarn_decode_workspace_bytes gives
 *     the need).  Allocates nothing and frees nothing.
 *   - The first call on each device looks up the array's device address with
 *     that device current; make that first call before any stream capture.
 *     The address is remembered per device and context: the first call after
 *     a cudaDeviceReset looks it up again, so it too should come before any
 *     stream capture.
 *   - Every call shares the one array and clears its ticket counters itself
 *     when its plan merges splits through them (a cudaMemsetAsync on
 *     `stream`, which allocates nothing);
 *     calls whose executions overlap on the GPU race on it, so serialise them
 *     (one stream, or events between streams). */
int kvarn_decode_attention_noalloc(const kvarn_config_t *cfg, const void *q, const void *pool,
                                   int64_t num_pages, const int32_t *block_table,
                                   int max_blocks, const int32_t *seq_lens, int batch,
                                   int max_seq, const void *tail_k, const void *tail_v,
                                   float softmax_scale, void *out, int32_t *status,
                                   kvarn_stream_t stream);

/* Chunked prefill: attention of a chunk of new query tokens per sequence over
 * the quantized cache ("KV Cache Nasil Calisir?": each token attends to every
 * cached token up to its own position; "Paged Attention (vLLM)" for the
 * pages).  Sequence b holds start[b] tokens before the chunk and chunk_lens[b]
 * new ones, and the cache (pool pages + fp16 tails) is already in its state
 * after the chunk was appended: n_b = start[b] + chunk_lens[b] tokens, the
 * n_b / 128 full blocks in the pool (block_table) and the n_b mod 128 newest
 * tokens in the tails (as kvarn_quantize_blocks leaves a sequence of length
 * n_b).  Query token i < chunk_lens[b] sits at position P = start[b] + i:
 *   out[b][i][h] = sum_{t <= P} softmax_t(scale * q[b][i][h] . k_t) v_t,
 * query head h reading KV head h / (Hq/Hkv); keys and values are dequantized
 * and rotated back as in kvarn_decode_attention.
 *   q, out      fp16 [batch][chunk_max][Hq][128]; rows i >= chunk_lens[b] of
 *               out are written as zeros
 *   start, chunk_lens  int32 [batch] (device); 0 <= chunk_lens[b] <= chunk_max
 *               and start[b] + chunk_lens[b] <= max_seq, else the sequence is
 *               reported (KVARN_STATUS_BAD_LENGTH) and its rows are zeros
 *   max_seq     host upper bound on start + chunk_lens
 * No workspace.  A page id outside the pool is reported
 * (KVARN_STATUS_BAD_PAGE) and the query tiles that would read it give zeros.
 * The work is one CTA per 128 query rows (128 / (Hq/Hkv) tokens of one KV
 * head's query group) and KV head; it uses up to 227 KB of shared memory and
 * 256 TMEM columns, so one CTA runs per SM.  Every record format is taken;
 * the 15360-byte (and smaller) records stream two pages ahead, the larger
 * ones ("k4v2_g64", "k4v4_g128", "k8v4_g128") one page at a time. */
int kvarn_chunk_attention(const kvarn_config_t *cfg, const void *q, int chunk_max,
                          const int32_t *start, const int32_t *chunk_lens, int batch,
                          int max_seq, const void *pool, int64_t num_pages,
                          const int32_t *block_table, int max_blocks, const void *tail_k,
                          const void *tail_v, float softmax_scale, void *out, int32_t *status,
                          kvarn_stream_t stream);

/* ---- SnapKV-style one-shot selection at the end of prefill ----
 * "Makale Bulteni - SnapKV" (cmlonder.com): the attention of the prompt's last
 * `window` tokens (the observation window, 32 or 64 on the page) over the
 * earlier tokens is scanned once, and each KV head keeps its most critical,
 * clustered positions; decode then runs on a compact cache of `capacity`
 * tokens per head (kvarn_snapkv_gather, then kvarn_quantize_blocks).
 * Readings: votes[b][h][t] = sum over the window queries (position
 * n - window + i) and the query heads of KV head h's group of their softmax
 * (over each query's causal context, scale softmax_scale) at prefix position
 * t < n - window; clustering = max pooling of the votes with the odd kernel
 * pool_kernel (window [t - k/2, t + k/2] clipped to the prefix); kept = the
 * capacity - window prefix positions with the largest pooled votes (ties to
 * the lower position), then the window, in increasing order; a prompt whose
 * prefix is no longer than capacity - window is kept whole. */

/* Workspace of kvarn_snapkv_select (16-byte aligned). */
size_t kvarn_snapkv_workspace_bytes(const kvarn_config_t *cfg, int batch, int window,
                                    int max_seq);

/*   q_window   fp16 [batch][window][Hq][128] (device), the queries of each
 *              prompt's last `window` tokens (row i = position n - window + i)
 *   k          fp16 (device), element (b, t, h, c) at b*stride_b + t*stride_t +
 *              h*stride_h + c (strides in elements, multiples of 8), t < max_seq
 *   seq_lens   int32 [batch] (device) prompt lengths n, window included
 *   capacity   tokens kept per (sequence, KV head), >= window
 *   pool_kernel odd pooling width >= 1
 *   votes      float32 [batch][Hkv][max_seq] (device), written whole (0 from
 *              n - window on)
 *   indices    int32 [batch][Hkv][capacity] (device): kept positions,
 *              increasing; -1 past the end of a prompt shorter than capacity
 *   workspace  kvarn_snapkv_workspace_bytes() bytes (device, 16-byte aligned;
 *              caller-owned, no contents kept between calls)
 * Three launches on `stream`: the window's scores on the tensor cores
 * (statistics, then votes), then pooling and selection.  A length outside
 * [0, max_seq] is reported (KVARN_STATUS_BAD_LENGTH) and that sequence treated
 * as empty; a wait that runs out is reported (KVARN_STATUS_TIMEOUT).
 * Returns KVARN_ERR_INVALID_ARG for null or misaligned pointers, bad strides,
 * window <= 0, capacity < window or an even kernel; KVARN_ERR_WORKSPACE for a
 * short workspace. */
int kvarn_snapkv_select(const kvarn_config_t *cfg, const void *q_window, int window,
                        const void *k, int64_t stride_b, int64_t stride_t, int64_t stride_h,
                        const int32_t *seq_lens, int batch, int max_seq, int capacity,
                        int pool_kernel, float softmax_scale, float *votes, int32_t *indices,
                        void *workspace, size_t workspace_bytes, int32_t *status,
                        kvarn_stream_t stream);

/* The kept tokens into the compact cache: k_out, v_out fp16
 * [batch][capacity][Hkv][128] (device, dense), token j of head h = token
 * indices[b][h][j] of k, v (same layout and strides as in
 * kvarn_snapkv_select, t < max_seq); a position outside [0, max_seq) (the -1
 * padding) gives zeros.  One launch on `stream`. */
int kvarn_snapkv_gather(const void *k, const void *v, int64_t stride_b, int64_t stride_t,
                        int64_t stride_h, int batch, int max_seq, int num_kv_heads,
                        const int32_t *indices, int capacity, void *k_out, void *v_out,
                        kvarn_stream_t stream);

/* Diagnosis: dequantizes `n` page records of the fp32-metadata format into
 * float32 rotated-space tiles.
 *   records   [n][15360] bytes (e.g. pool + page*Hkv*15360, one record per
 *             (page, head) in order)
 *   yk, yv    float32 [n][128 tokens][128 channels]:
 *             yhat_td = c_d * (s'_t * q_td + z'_t) */
int kvarn_dequantize_pages(const void *records, int64_t n, float *yk, float *yv,
                           kvarn_stream_t stream);

/* Diagnosis for every record format: dequantizes `n` page records of the
 * format `cfg` names ("KVarN Nasil Calisir?", the inverse of stage
 * "Kuantize Edilmis Onbellek") into float32 rotated-space tiles.
 *   records   [n][kvarn_page_bytes(cfg)] bytes, 16-byte aligned (device)
 *   yk, yv    float32 [n][128 tokens][128 channels] (device), written:
 *             yhat_td = alpha_t beta_d q_td + gamma_t delta_d, with
 *             (alpha, gamma) = (s', z') of the token (of the channel's
 *             group for groups of 64) and beta = delta = c_d, or for "_pc"
 *             alpha = gamma = r_t and (beta, delta) = (cs_d, cz_d); fp16
 *             metadata ("_m16") is widened to fp32 first.
 * Returns KVARN_ERR_UNSUPPORTED for a bad config, KVARN_ERR_INVALID_ARG for
 * n < 0, a null or misaligned pointer; one launch on `stream`. */
int kvarn_dequantize_records(const kvarn_config_t *cfg, const void *records, int64_t n,
                             float *yk, float *yv, kvarn_stream_t stream);

/* Diagnosis of the bounded waits: every wait of the library's kernels on an
 * mbarrier (a bulk copy landing, an MMA completing, a peer warp's arrival)
 * gives up after a time limit, reports KVARN_STATUS_TIMEOUT and lets the
 * kernel end, instead of hanging the GPU.  This call runs that same wait in
 * a one-warp kernel on a barrier of its own that receives its one arrival
 * first (arrive = 1: no timeout) or never (arrive = 0: the wait runs out
 * after limit_us microseconds and KVARN_STATUS_TIMEOUT is OR-ed into
 * *status).  status: device int32, not null; limit_us in [1, 1000000].
 * Returns KVARN_ERR_INVALID_ARG for bad arguments; one launch on `stream`. */
int kvarn_wait_check(int32_t *status, int arrive, uint32_t limit_us, kvarn_stream_t stream);

/* ---- The FP16 paged cache the quantized one is measured against ----
 * The KVarN page (blog.edumints.com) states its capacity and throughput gains
 * relative to an FP16 KV cache; these calls are that baseline on the same
 * harness: the same block table and lengths, every token kept as fp16.
 * Page: one per (page, KV head), KVARN_FP16_PAGE_BYTES bytes, 16-byte aligned:
 *   [0, 32768)      K, [128 tokens][128 channels] fp16
 *   [32768, 65536)  V, same
 * Pool = [num_pages][num_kv_heads][KVARN_FP16_PAGE_BYTES].  Block j of a
 * sequence holds its tokens 128j .. 128j + 127; the last block is filled up
 * to the length and the rest of it is never read. */
#define KVARN_FP16_PAGE_BYTES 65536

/* Copies tokens [0, seq_lens[b]) of every sequence into its fp16 pages.
 *   k, v       fp16, element (b, t, h, c) at b*stride_b + t*stride_t +
 *              h*stride_h + c (strides in elements, multiples of 8)
 *   seq_lens   int32 [batch] (device), 0 <= len <= max_seq
 *   block_table int32 [batch][max_blocks] (device); every block holding a
 *              token must be in the table (max_blocks >= ceil(max_seq/128))
 * Bad page ids and lengths are reported in *status and skipped. */
int kvarn_fp16_write_blocks(const void *k, const void *v, int64_t stride_b, int64_t stride_t,
                            int64_t stride_h, int batch, int num_kv_heads,
                            const int32_t *seq_lens, int max_seq, const int32_t *block_table,
                            int max_blocks, void *pool, int64_t num_pages, int32_t *status,
                            kvarn_stream_t stream);

/* Bytes of workspace kvarn_fp16_decode_attention needs on the current device
 * (0: none, or no CUDA device is current). */
size_t kvarn_fp16_decode_workspace_bytes(int num_q_heads, int num_kv_heads, int batch,
                                         int max_seq);

/* Decode attention over the fp16 pages, one query token per sequence:
 *   out[b][h] = sum_t softmax_t(scale * q[b][h] . k_t) v_t, t < seq_lens[b]
 * Query head h reads KV head h / (Hq/Hkv); Hq/Hkv at most 8.  Arguments as
 * for kvarn_decode_attention (q, out fp16 [batch][Hq][128]; the workspace
 * zero-filled before its first use and left so).  Split-K over the pages with
 * a log-sum-exp merge in the same launch. */
int kvarn_fp16_decode_attention(const void *q, int num_q_heads, int num_kv_heads,
                                const void *pool, int64_t num_pages, const int32_t *block_table,
                                int max_blocks, const int32_t *seq_lens, int batch, int max_seq,
                                float softmax_scale, void *out, void *workspace,
                                size_t workspace_bytes, int32_t *status, kvarn_stream_t stream);

/* ---- The FP8 paged cache, the second baseline ----
 * The glossary "KV Cache (Anahtar-Deger Onbellegi)" (yapayzekasozluk.tr),
 * "Sik Sorulan Sorular", names INT8/FP8 KV quantization as the common way to
 * halve the cache; these calls are that cache on the same harness.  Each
 * token of each KV head is stored as e4m3 codes (largest finite 448) with one
 * fp32 scale s = max|x| / 448: codes = e4m3(x / s), nearest even, saturated;
 * both divisions fp32.  Page: one per (page, KV head), KVARN_FP8_PAGE_BYTES
 * bytes, 16-byte aligned:
 *   [0, 16384)      K codes [128 tokens][128 channels]
 *   [16384, 32768)  V codes, same
 *   [32768, 33280)  K scales fp32 [128 tokens]
 *   [33280, 33792)  V scales fp32 [128 tokens]
 * Pool = [num_pages][num_kv_heads][KVARN_FP8_PAGE_BYTES]; 264 bytes per
 * token-head against 512 in fp16.  The calls take the arguments of the
 * kvarn_fp16_* calls above, with this page layout. */
#define KVARN_FP8_PAGE_BYTES 33792

/* Quantizes tokens [0, seq_lens[b]) of every sequence into its fp8 pages. */
int kvarn_fp8_write_blocks(const void *k, const void *v, int64_t stride_b, int64_t stride_t,
                           int64_t stride_h, int batch, int num_kv_heads,
                           const int32_t *seq_lens, int max_seq, const int32_t *block_table,
                           int max_blocks, void *pool, int64_t num_pages, int32_t *status,
                           kvarn_stream_t stream);

/* Bytes of workspace kvarn_fp8_decode_attention needs on the current device
 * (0: none, or no CUDA device is current). */
size_t kvarn_fp8_decode_workspace_bytes(int num_q_heads, int num_kv_heads, int batch,
                                        int max_seq);

/* Decode attention over the fp8 pages, one query token per sequence:
 *   out[b][h] = sum_t softmax_t(scale * q[b][h] . k_t) v_t, t < seq_lens[b],
 * k_t = s^K_t e4m3(K codes), v_t likewise; Hq/Hkv at most 8; split-K with a
 * log-sum-exp merge in the same launch, the workspace as for the FP16 call. */
int kvarn_fp8_decode_attention(const void *q, int num_q_heads, int num_kv_heads,
                               const void *pool, int64_t num_pages, const int32_t *block_table,
                               int max_blocks, const int32_t *seq_lens, int batch, int max_seq,
                               float softmax_scale, void *out, void *workspace,
                               size_t workspace_bytes, int32_t *status, kvarn_stream_t stream);

/* Static text for a return code or a status bit set. */
const char *kvarn_status_string(int code);

/* Library version, "major.minor.patch". */
const char *kvarn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVARN_H */
