/* NVFP4 KV cache for GB300 (sm_103a): fused quantize-append and paged GQA attention.
 *
 * C ABI. Every pointer is a plain host or device pointer as stated per argument; no framework
 * types cross this boundary. CUDA streams are passed as `void *` holding a cudaStream_t
 * (NULL = the legacy default stream). All device work is asynchronous on that stream.
 *
 * Method sources (web pages, cited by address and section):
 *   [NVFP4] prismix.dev/news/833001997676, section "NVFP4 KV cache (from scratch)":
 *           4-bit E2M1 codes with one E4M3 scale per 16 elements for K and V, scales in natural
 *           row-major order, a Hadamard rotation of K (and Q) before quantisation, V unrotated,
 *           Q and K both quantised for the Q.K^T product, V dequantised for P.V, the current
 *           token's K/V quantised in the decode path with no separate pass, and 144 bytes per
 *           token per KV head.
 *   [YaRN]  same page, section "YaRN context extension": theta = 1e7, 25 % of the head dims
 *           rotary, linear position scaling.
 *
 * Data layout (caller-allocated device memory, 16-byte aligned):
 *   Pool: num_pages blocks of kv_nvfp4_page_bytes() = num_kv_heads * 9216 bytes, one block per
 *   page of 64 token slots holding every KV head. Within a block (H = num_kv_heads):
 *     [0, 4096 H)          K codes, head h at 4096 h, in the tensor-core tile order: byte j
 *                          (0..63) of slot k sits at (k / 8) * 512 + (j / 16) * 128 +
 *                          (k % 8) * 16 + (j % 16), i.e. 8-slot x 16-byte core tiles
 *     [4096 H, 4608 H)     K scales, in the order the tensor core's scale-factor copy reads them:
 *                          scale b of slot k of head h is at 4096 H + 1024 (h / 2) + 512 c
 *                          + 16 (k % 32) + 8 (h % 2) + 4 (k / 32) + b % 4 with c = b / 4, or,
 *                          for a last head without a partner (odd H), at 4096 H + 1024 (h / 2)
 *                          + 256 c + 8 (k % 32) + 4 (k / 32) + b % 4
 *     [4608 H, 8704 H)     V codes, head h at 4608 H + 4096 h: slot k at 64 k (row-major)
 *     [8704 H, 9216 H)     V scales, head h at 8704 H + 512 h: slot k at 8 k (row-major)
 *   A 64-byte code row holds 128 E2M1 codes: element 2j in the low nibble of byte j, element
 *   2j+1 in the high nibble. A scale row holds 8 E4M3 scales; scale b covers elements
 *   16b..16b+15. => 64 + 8 bytes for K and again for V: 144 bytes per token per KV head.
 *   Token `pos` of sequence `s` lives in page block_table[s * max_pages + pos / 64], slot
 *   pos % 64. K rows are stored after RoPE and the normalised Hadamard rotation; V rows raw.
 *   Quantised Q: q_codes [tokens][num_q_heads][64] (row-major), q_scales
 *   [tokens][num_q_heads][8], after RoPE and rotation, in the same encoding.
 *
 * Ownership: the caller allocates and frees every device buffer. No entry point allocates
 * device memory. A plan workspace belongs to the stream it was planned on: reuse or overwrite
 * it only after the attention call that reads it has completed on that stream, and do not run
 * two attention calls with the same workspace concurrently.
 *
 * Errors: every entry point returns a kv_nvfp4_status. Host-checkable faults return
 * KV_NVFP4_EINVAL before any launch. Launch failures return KV_NVFP4_ECUDA. Data-dependent
 * faults found on the device (a page id outside the pool, a position beyond the page table or
 * the RoPE table, a sequence id out of range) set bits (KV_NVFP4_DEV_*) in the caller's int32
 * `d_status` word with an atomic OR, and the offending row or page is skipped; pass NULL to
 * ignore them. The library never traps and never spins without a bound.
 */
#ifndef KV_NVFP4_H
#define KV_NVFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t kv_nvfp4_status;
#define KV_NVFP4_OK 0
#define KV_NVFP4_EINVAL (-1)
#define KV_NVFP4_ECUDA (-2)
#define KV_NVFP4_ENOSPACE (-3)

/* Bits written to *d_status by device code. */
#define KV_NVFP4_DEV_BAD_PAGE 0x1     /* block_table entry outside [0, num_pages) */
#define KV_NVFP4_DEV_BAD_POS 0x2      /* position < 0 or >= max_pages * 64 */
#define KV_NVFP4_DEV_BAD_SEQ 0x4      /* sequence id outside [0, num_seqs) */
#define KV_NVFP4_DEV_BAD_ROPE 0x8     /* position >= rope_max_pos for a rotated row */
#define KV_NVFP4_DEV_TIMEOUT 0x10     /* an internal barrier wait hit its time limit */

/* Model geometry of one attention layer. The library supports head_dim = 128 and
 * page_size = 64; num_q_heads (at most 4096) must be a multiple of num_kv_heads; rot_dim is a
 * multiple of 8 and at most 128 (0 disables RoPE). */
typedef struct kv_nvfp4_layout {
  int32_t num_q_heads;  /* 24 in the pages' model */
  int32_t num_kv_heads; /* 4 */
  int32_t head_dim;     /* 128 */
  int32_t page_size;    /* 64 tokens */
  int32_t rot_dim;      /* 32 = 25 % of 128 [YaRN] */
} kv_nvfp4_layout;

/* Filled by kv_nvfp4_plan; passed unchanged to kv_nvfp4_decode_attn. A row is (query token, head
 * within the GQA group): row = token * group + head_in_group, group * q_len rows per KV head.
 * With at most 8 rows per KV head and at most 4 KV heads (decode) a group is one (sequence, tile
 * of 8 rows), covering every KV head; otherwise (speculative verify, prefill chunks, wider layouts)
 * a group is one (sequence, KV head, tile of 128 rows), run by the tile kernel. A group's pages
 * are split into chunks of chunk_pages pages, and the chunks of all groups are shared out over
 * `grid` CTAs in contiguous ranges (one range may hold several chunks of a group, which the CTA
 * combines as it goes): page-balanced for the decode kernel, and for the tile kernel balanced on
 * pages plus a fixed charge of ten pages per segment (the smallest per-CTA cap that `grid` CTAs
 * can fill, so trailing CTAs may get no work). */
typedef struct kv_nvfp4_plan_info {
  int32_t num_seqs;
  int32_t q_len;
  int32_t causal;          /* causal masking among the q_len new tokens (pages past the last
                              visible key of a row tile are not visited) */
  int32_t chunk_pages;     /* split-K granularity, in pages */
  int32_t num_kv_heads;
  int32_t num_row_groups;  /* row tiles per sequence: ceil(group * q_len / 8), or
                              ceil(group * q_len / 128) on the tile kernel */
  int32_t num_groups;      /* num_seqs * num_row_groups, times num_kv_heads on the tile kernel */
  int32_t num_segments;    /* contiguous (group, page range) pieces over all CTAs */
  int32_t num_partials;    /* partial-result slots (segments of groups split over CTAs) */
  int32_t grid;            /* CTAs of the attention launch, at most the SM count */
  int32_t max_seq_len;     /* longest sequence; must fit max_pages * 64 at attention time */
  int32_t num_split_groups; /* groups split over several CTAs (merged by a second launch) */
  int64_t total_kv_tokens; /* sum of seq_lens */
  int64_t total_pages;     /* pages visited by one attention call, summed over groups */
  uint64_t off_groups, off_segments, off_cta, off_split, off_partials; /* byte offsets */
  uint64_t workspace_bytes;
} kv_nvfp4_plan_info;

/* Human-readable name of a status code (static string). */
const char *kv_nvfp4_status_string(kv_nvfp4_status status);

/* Description of the CUDA error behind this thread's most recent KV_NVFP4_ECUDA (static string). */
const char *kv_nvfp4_last_cuda_error(void);

/* Library version as major * 10000 + minor * 100 + patch. */
int32_t kv_nvfp4_version(void);

/* Validates a layout; KV_NVFP4_OK or KV_NVFP4_EINVAL. */
kv_nvfp4_status kv_nvfp4_layout_check(const kv_nvfp4_layout *layout);

/* Bytes of one pool page over all KV heads, K and V, codes and scales:
 * 64 * 144 * num_kv_heads (36,864 for 4 KV heads) [NVFP4]. 0 on an invalid layout. */
size_t kv_nvfp4_page_bytes(const kv_nvfp4_layout *layout);

/* Bytes of a pool of num_pages pages (num_pages * kv_nvfp4_page_bytes). */
kv_nvfp4_status kv_nvfp4_pool_bytes(const kv_nvfp4_layout *layout, int32_t num_pages,
                                    size_t *bytes);

/* ---- RoPE table [YaRN] ----------------------------------------------------------------------
 * fp32 table [max_pos][rot_dim]: entries 0..rot_dim/2-1 are cos, rot_dim/2..rot_dim-1 are sin,
 * of angle (pos / pos_scale) * theta^(-2i/rot_dim), evaluated in double on the host and rounded
 * once to fp32. Dimension i < rot_dim/2 rotates with dimension i + rot_dim/2. pos_scale is the
 * linear position-scaling factor (1 = none; 600000/262144 stretches a 262k model to 600k). */
size_t kv_nvfp4_rope_table_bytes(int32_t max_pos, int32_t rot_dim);

/* Fills a HOST buffer of kv_nvfp4_rope_table_bytes bytes. No CUDA call. */
kv_nvfp4_status kv_nvfp4_rope_table_fill_host(float *h_table, int32_t max_pos, int32_t rot_dim,
                                              double theta, double pos_scale);

/* Computes the table on the host and copies it into DEVICE memory d_table on `stream`. The
 * host staging copy is consumed before return. */
kv_nvfp4_status kv_nvfp4_rope_table_init(float *d_table, int32_t max_pos, int32_t rot_dim,
                                         double theta, double pos_scale, void *stream);

/* ---- Fused quantize-append [NVFP4: Hadamard rotation, quantisation, fused append] ---------
 * For each of T tokens: every Q head (if q != NULL) and every K head gets RoPE on its first
 * rot_dim dims, the normalised 128-point Walsh-Hadamard rotation (Sylvester order, stages
 * h = 1..64, then a multiply by fp32 rn(2^-3.5)), and NVFP4 quantisation; every V head gets the
 * quantisation only. Quantisation per 16 elements: scale = E4M3 round-to-nearest-even of
 * amax/6, saturating at 448; code = E2M1 round-to-nearest-even of x / scale, saturating at 6,
 * sign kept; a block whose scale is 0 stores zero codes. K/V rows go into their page slots,
 * Q rows into q_codes/q_scales at the token's index.
 *   q, k, v:        DEVICE bf16 [T][num_q_heads][128], [T][num_kv_heads][128] (q may be NULL,
 *                   then q_codes/q_scales are ignored)
 *   d_seq_ids:      DEVICE int32 [T], sequence of each token, in [0, num_seqs)
 *   d_positions:    DEVICE int32 [T], absolute position of each token in its sequence
 *   d_rope_table:   DEVICE fp32 table from kv_nvfp4_rope_table_init, rope_max_pos rows
 *   d_block_table:  DEVICE int32 [num_seqs][max_pages]
 *   pool:           DEVICE pool of num_pages pages (see layout above)
 *   q_codes/q_scales: DEVICE [T][num_q_heads][64] / [T][num_q_heads][8]
 *   d_status:       DEVICE int32 or NULL
 * One kernel launch. T = 0 is a no-op. */
kv_nvfp4_status kv_nvfp4_append(const kv_nvfp4_layout *layout, const void *q, const void *k,
                                const void *v, const int32_t *d_seq_ids,
                                const int32_t *d_positions, int32_t T, const float *d_rope_table,
                                int32_t rope_max_pos, const int32_t *d_block_table,
                                int32_t num_seqs, int32_t max_pages, int32_t num_pages,
                                uint8_t *pool, uint8_t *q_codes, uint8_t *q_scales,
                                int32_t *d_status, void *stream);

/* ---- Page-table / split-K setup ------------------------------------------------------------
 * Sizes and builds the work list of one attention call from HOST sequence lengths (after the
 * append, i.e. including the q_len new tokens). chunk_tokens (a positive multiple of 64) is the
 * split-K granularity: a sequence is only ever cut between chunks. 1024 suits long-context
 * decode; 64 lets the plan balance the CTAs to the page. The workspace holds the group and
 * segment tables, the list of split groups (those that span more than one CTA), and one
 * (m, l, O) partial per segment of every split group: 4160 bytes per KV head for 8-row tiles,
 * 66,560 bytes for the tile kernel's 128-row tiles. */
kv_nvfp4_status kv_nvfp4_plan_workspace_bytes(const kv_nvfp4_layout *layout,
                                              const int32_t *h_seq_lens, int32_t num_seqs,
                                              int32_t q_len, int32_t causal,
                                              int32_t chunk_tokens, size_t *bytes);

/* Host-only variant of kv_nvfp4_plan for a given CTA count: writes the image of the workspace
 * tables (groups, segments, per-CTA segment ranges, split-group list; everything before
 * info->off_partials) into HOST memory h_workspace and fills *info. No CUDA call. Layout of the
 * image: groups are 8 int32 {seq, pair, row_tile, seq_len, n_segments, first_partial, pages, 0}
 * (pair = 0 for 8-row tiles, which cover every KV head);
 * segments are 4 int32 {group, page_lo, page_hi, partial or -1}; CTA b owns segments
 * [cta[b], cta[b+1]); the split list holds info->num_split_groups group indices in order. */
kv_nvfp4_status kv_nvfp4_plan_host(const kv_nvfp4_layout *layout, const int32_t *h_seq_lens,
                                   int32_t num_seqs, int32_t q_len, int32_t causal,
                                   int32_t chunk_tokens, int32_t num_ctas, void *h_workspace,
                                   size_t ws_bytes, kv_nvfp4_plan_info *info);

/* Writes the work list into DEVICE memory d_workspace (ws_bytes at least the size above) on
 * `stream` (one host-to-device copy) and fills *info (HOST). Every seq_len must be >= q_len
 * and >= 1. The CTA count is taken from the current device's SM count. The workspace holds
 * one (m, l, O) partial per segment of a group spread over several CTAs (sizes above). */
kv_nvfp4_status kv_nvfp4_plan(const kv_nvfp4_layout *layout, const int32_t *h_seq_lens,
                              int32_t num_seqs, int32_t q_len, int32_t causal,
                              int32_t chunk_tokens, void *d_workspace, size_t ws_bytes,
                              kv_nvfp4_plan_info *info, void *stream);

/* ---- Paged GQA decode / speculative-verify attention [NVFP4: NVFP4 Q.K^T, V dequantised]
 * For every sequence s and each of its q_len query tokens i (position seq_len - q_len + i) and
 * every query head h (kv head h / (num_q_heads / num_kv_heads)):
 *   out = sum_t softmax_t(sm_scale * qhat . khat_t) * vhat_t
 * over keys t < seq_len, restricted to t <= seq_len - q_len + i when the plan is causal, where qhat,
 * khat, vhat are the dequantised NVFP4 rows (code value times block scale). Scores and the
 * softmax run in fp32 with split-K over the plan's chunks.
 *   plan, d_workspace: from kv_nvfp4_plan (same stream)
 *   q_codes/q_scales: DEVICE [num_seqs * q_len][num_q_heads][64 | 8], sequence-major
 *   sm_scale:       softmax scale; <= 0 selects 1/sqrt(head_dim)
 *   pool, num_pages, d_block_table, max_pages: as for kv_nvfp4_append
 *   out:            DEVICE fp32 [num_seqs * q_len][num_q_heads][128]
 * Two kernel launches on `stream`: the attention kernel (one persistent CTA per SM), then, when
 * the plan has split groups, the merge of their partials (one CTA per split group, KV head and
 * row). With at most 8 rows per KV head and at most 4 KV heads the attention kernel is the decode
 * kernel (every head of a page staged together; Q.K^T block-scaled on the tensor cores, P.V on the
 * warp-level tensor path); otherwise it is the tile kernel (128 rows of one KV head per tile, keys
 * in blocks of 128; Q.K^T block-scaled and P.V in f16 with P in tensor memory, both on the tcgen05
 * tensor cores, O accumulated in tensor memory), which takes any number of KV heads and any group
 * size. The workspace may be
 * reused by the next call on the same stream; calls that overlap on one workspace race. */
kv_nvfp4_status kv_nvfp4_decode_attn(const kv_nvfp4_layout *layout,
                                     const kv_nvfp4_plan_info *plan, void *d_workspace,
                                     const uint8_t *q_codes, const uint8_t *q_scales,
                                     float sm_scale, const uint8_t *pool, int32_t num_pages,
                                     const int32_t *d_block_table, int32_t max_pages, float *out,
                                     int32_t *d_status, void *stream);

/* ---- Fused decode step [NVFP4: the decode path quantises the current K/V as it runs] -----------
 * One launch doing what kv_nvfp4_append (of the step's new tokens, with Q) followed by
 * kv_nvfp4_decode_attn does, with bit-identical pool bytes and output: the new tokens are encoded
 * (RoPE, Hadamard rotation, NVFP4) inside the attention kernel, the K/V rows stored into the pool
 * by the CTA that reads their page, and the Q rows used straight from shared memory.
 *   plan, d_workspace: from kv_nvfp4_plan over the lengths INCLUDING the new tokens (same stream)
 *   q, k, v:   DEVICE bf16 [num_seqs * q_len][num_q_heads | num_kv_heads][128], sequence-major:
 *              row s * q_len + i is new token i of sequence s, at position seq_len_s - q_len + i
 *   d_rope_table, rope_max_pos, d_block_table, max_pages, num_pages, pool: as for the append
 *   q_codes_out, q_scales_out: optional (both or neither) DEVICE copy of the encoded Q rows,
 *              [num_seqs * q_len][num_q_heads][64 | 8] (q_codes_out 16-byte aligned, else EINVAL)
 *   sm_scale, out, d_status: as for kv_nvfp4_decode_attn
 * Requires (num_q_heads / num_kv_heads) * q_len <= 8 and num_kv_heads <= 4 (one 8-row tile per
 * sequence on the decode kernel: decode with GQA groups up to 8); larger verify or prefill steps,
 * wider groups and more KV heads use the two calls. Status bits as for both
 * calls (a bad page or position skips the row). One kernel launch, plus the split-K merge launch
 * when the plan has split groups. */
kv_nvfp4_status kv_nvfp4_decode_step(const kv_nvfp4_layout *layout,
                                     const kv_nvfp4_plan_info *plan, void *d_workspace,
                                     const void *q, const void *k, const void *v,
                                     const float *d_rope_table, int32_t rope_max_pos,
                                     const int32_t *d_block_table, int32_t max_pages,
                                     int32_t num_pages, uint8_t *pool, uint8_t *q_codes_out,
                                     uint8_t *q_scales_out, float sm_scale, float *out,
                                     int32_t *d_status, void *stream);

/* ---- One decode step from host buffers ------------------------------------------------------
 * No counterpart in the pages: kv_nvfp4_plan followed by kv_nvfp4_decode_step, with the step's
 * new tokens and its output in HOST memory, enqueued on `stream` by one call: the host-to-device
 * copies of q, k and v into the caller's device buffers, the plan build and its upload, the
 * fused step's launches, and the device-to-host copy of the output. For a serving loop that
 * drives the library from host code once per step.
 *   h_seq_lens, num_seqs, q_len, causal, chunk_tokens: as for kv_nvfp4_plan (HOST lengths
 *              including the new tokens); (num_q_heads / num_kv_heads) * q_len <= 8 and
 *              num_kv_heads <= 4
 *   d_workspace, ws_bytes: at least kv_nvfp4_plan_workspace_bytes bytes (DEVICE, 16-byte aligned)
 *   h_q, h_k, h_v: HOST bf16 rows laid out as q, k, v of kv_nvfp4_decode_step; keep them
 *              unchanged until the stream has passed this call's work
 *   d_q, d_k, d_v: DEVICE buffers of the same sizes (16-byte aligned) that receive them
 *   d_rope_table, rope_max_pos, d_block_table, max_pages, num_pages, pool, sm_scale, d_status:
 *              as for kv_nvfp4_decode_step
 *   d_out:     DEVICE fp32 buffer [num_seqs * q_len][num_q_heads][128]
 *   h_out:     HOST fp32 output of the same shape, complete when the stream reaches the end of
 *              this call's work
 *   plan_out:  optional HOST copy of the plan info (may be null)
 * When h_q, h_k, h_v and h_out are page-locked and 16-byte aligned, no copy-engine operation is
 * enqueued: a small kernel reads the new rows over the host link into d_q, d_k, d_v and writes
 * the work list (passed inline when it is at most 8 KB, else copied), and the attention and merge
 * kernels write the output rows straight into h_out (d_out is not written). Otherwise the rows and
 * the work list are copied in, the output goes to d_out and is copied to h_out (pageable memory is
 * staged by the runtime, which may wait for the stream's earlier work).
 * Returns once everything is enqueued; EINVAL before any copy for the argument checks above, or
 * the first error of the calls it makes. */
kv_nvfp4_status kv_nvfp4_decode_step_host(
    const kv_nvfp4_layout *layout, const int32_t *h_seq_lens, int32_t num_seqs, int32_t q_len,
    int32_t causal, int32_t chunk_tokens, void *d_workspace, size_t ws_bytes, const void *h_q,
    const void *h_k, const void *h_v, void *d_q, void *d_k, void *d_v, const float *d_rope_table,
    int32_t rope_max_pos, const int32_t *d_block_table, int32_t max_pages, int32_t num_pages,
    uint8_t *pool, float sm_scale, float *d_out, float *h_out, int32_t *d_status,
    kv_nvfp4_plan_info *plan_out, void *stream);

/* ---- Comparator KV formats [NVFP4 "Result": 144 B per token per KV head vs 264 int8 vs 512 bf16;
 * upstream NVFP4 K with fp16 V and no rotation] -------------------------------------------------
 * prismix.dev/news/833001997676, section "NVFP4 KV cache (from scratch)". Decode attention over
 * three other KV formats, for byte-count and roofline comparison with the NVFP4 path; not the
 * method itself. Q is unquantised in all three (bf16 after RoPE).
 *   KV_CMP_BF16:  K = bf16(RoPE(k)), V = v                                   512 B/token/KV head
 *   KV_CMP_INT8:  per row (K after RoPE, V raw) s = amax / 127 (fp32), codes = RNE(x / s)
 *                 clamped to +-127, s stored as fp32                          264 B
 *   KV_CMP_K4V16: K = NVFP4 of RoPE(k) without the Hadamard rotation, V = fp16(v)   328 B
 * Pool: num_pages blocks of kv_cmp_page_bytes; a block holds one chunk per KV head (K rows, then
 * V rows, of its 64 slots; the chunk layouts and the 16-byte unit swizzle inside rows are given
 * in bit_kv_cache_03_gb300/csrc/compare.cu). */
#define KV_CMP_BF16 0
#define KV_CMP_INT8 1
#define KV_CMP_K4V16 2

/* Bytes of one comparator page (all KV heads); 0 for an invalid layout or format. */
size_t kv_cmp_page_bytes(const kv_nvfp4_layout *layout, int32_t fmt);

/* Comparator append: as kv_nvfp4_append (same ids, positions, RoPE table, block table, status
 * bits and errors), writing K/V rows in format `fmt` and, when q is given, the bf16 RoPE'd Q rows
 * to q_out (DEVICE bf16 [T][num_q_heads][128], 16-byte aligned). One kernel launch. */
kv_nvfp4_status kv_cmp_append(const kv_nvfp4_layout *layout, int32_t fmt, const void *q,
                              const void *k, const void *v, const int32_t *d_seq_ids,
                              const int32_t *d_positions, int32_t T, const float *d_rope_table,
                              int32_t rope_max_pos, const int32_t *d_block_table,
                              int32_t num_seqs, int32_t max_pages, int32_t num_pages,
                              uint8_t *pool, void *q_out, int32_t *d_status, void *stream);

/* Plan for the comparator decode: as kv_nvfp4_plan, for (SM count / num_kv_heads) CTAs, each of
 * which the decode launches once per KV head. */
kv_nvfp4_status kv_cmp_plan_workspace_bytes(const kv_nvfp4_layout *layout,
                                            const int32_t *h_seq_lens, int32_t num_seqs,
                                            int32_t q_len, int32_t causal, int32_t chunk_tokens,
                                            size_t *bytes);
kv_nvfp4_status kv_cmp_plan(const kv_nvfp4_layout *layout, const int32_t *h_seq_lens,
                            int32_t num_seqs, int32_t q_len, int32_t causal, int32_t chunk_tokens,
                            void *d_workspace, size_t ws_bytes, kv_nvfp4_plan_info *plan,
                            void *stream);

/* Comparator decode attention over a pool of format `fmt`: q_rot = the q_out rows of
 * kv_cmp_append (num_seqs * q_len tokens, sequence-major); plan and workspace from kv_cmp_plan;
 * out, d_status, sm_scale and the errors as for kv_nvfp4_decode_attn. One kernel launch, plus
 * the split-K merge launch when the plan has split groups. */
kv_nvfp4_status kv_cmp_decode_attn(const kv_nvfp4_layout *layout, int32_t fmt,
                                   const kv_nvfp4_plan_info *plan, void *d_workspace,
                                   const void *q_rot, float sm_scale, const uint8_t *pool,
                                   int32_t num_pages, const int32_t *d_block_table,
                                   int32_t max_pages, float *out, int32_t *d_status,
                                   void *stream);

/* ---- Page spill and restore [Spill: cache pages moved out to host memory and back] ----------
 * prismix.dev/news/833001997676, section "Multi-level prefix reuse with host-KV safety net".
 * kv_nvfp4_spill_pages:   arena slot i <- pool page d_page_ids[i], for i < n
 * kv_nvfp4_restore_pages: pool page d_page_ids[i] <- arena slot i
 * A page block (kv_nvfp4_page_bytes: every KV head's K and V codes and scales of 64 slots) is
 * self-contained, so a page moves as one byte copy; a restored page may take another page id than
 * it had, with the block table renamed to match.
 *   pool:        DEVICE, num_pages page blocks (kv_nvfp4_pool_bytes), 16-byte aligned
 *   d_page_ids:  DEVICE int32 [n]; an id outside [0, num_pages) sets KV_NVFP4_DEV_BAD_PAGE and its
 *                copy is skipped (the arena slot, or the pool page, is left as it was). Restore
 *                ids should be distinct: a repeated id leaves that page holding one of its slots.
 *   arena:       n * kv_nvfp4_page_bytes bytes, 16-byte aligned, in memory the GPU can address:
 *                page-locked host memory (cudaHostAlloc, cudaMallocHost, cudaHostRegister: the
 *                GPU's own loads and stores reach it over the host link) or device memory.
 *                Pageable host memory is refused with KV_NVFP4_EINVAL.
 * One kernel launch on `stream`, asynchronous: the caller keeps pool, ids and arena alive, and
 * does not touch the arena's slots, until the stream has passed the call. n = 0 does nothing.
 * EINVAL for a bad layout, n < 0, a null or misaligned buffer, or num_pages <= 0. */
kv_nvfp4_status kv_nvfp4_spill_pages(const kv_nvfp4_layout *layout, const uint8_t *pool,
                                     int32_t num_pages, const int32_t *d_page_ids, int32_t n,
                                     uint8_t *arena, int32_t *d_status, void *stream);
kv_nvfp4_status kv_nvfp4_restore_pages(const kv_nvfp4_layout *layout, const uint8_t *arena,
                                       const int32_t *d_page_ids, int32_t n, uint8_t *pool,
                                       int32_t num_pages, int32_t *d_status, void *stream);

/* ---- Decode attention without caller-provided device memory ----------------------------------
 * No counterpart in the pages: an addition of this library for callers that cannot allocate
 * device memory, such as an inference engine that reserves all of the GPU's memory for its own
 * arena at start-up and passes a layer only its inputs and outputs, or a plug-in running under an
 * allocator it does not control, where cudaMalloc fails or stalls every stream on the device.
 *
 * Same result as kv_nvfp4_plan followed by kv_nvfp4_decode_attn (same arguments, same kernels),
 * but the workspace is a fixed buffer of KV_NVFP4_NOALLOC_SCRATCH_BYTES inside the library, held
 * on every GPU that loads the library until the process exits; nothing is allocated on the device.
 *   h_seq_lens, num_seqs, q_len, causal, chunk_tokens: as for kv_nvfp4_plan (HOST lengths)
 *   the rest: as for kv_nvfp4_decode_attn
 * Returns KV_NVFP4_ENOSPACE, before any GPU work, when the plan's workspace
 * (kv_nvfp4_plan_workspace_bytes) exceeds the buffer; callers then use the workspace path.
 * The first call on a device (in each of its contexts) looks up the buffer's device address with
 * that device current and keeps it for the later calls. Each call builds its work list in host
 * memory and uploads it, so the call cannot be recorded into a CUDA graph: while `stream` is
 * capturing it returns KV_NVFP4_EINVAL before enqueuing anything. Every call shares the buffer:
 * each rewrites its work list before its kernels read it and nothing in it has to start at zero,
 * but calls whose kernels overlap on the GPU (other streams, other host threads) corrupt each
 * other's results and must be serialised by the caller. */
#define KV_NVFP4_NOALLOC_SCRATCH_BYTES (32u << 20)

kv_nvfp4_status kv_nvfp4_decode_attn_noalloc(const kv_nvfp4_layout *layout,
                                             const int32_t *h_seq_lens, int32_t num_seqs,
                                             int32_t q_len, int32_t causal, int32_t chunk_tokens,
                                             const uint8_t *q_codes, const uint8_t *q_scales,
                                             float sm_scale, const uint8_t *pool,
                                             int32_t num_pages, const int32_t *d_block_table,
                                             int32_t max_pages, float *out, int32_t *d_status,
                                             void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KV_NVFP4_H */
