/*
 * mla.h — C ABI of the absorbed Multi-head Latent Attention decode library
 * (libmla.so, GB300 / sm_103a).
 *
 * What it computes.  One decode step of DeepSeek MLA in absorbed form over a
 * paged latent KV cache:
 *   q_lat[b,h,:] = W_UK[h]^T q_nope[b,h,:]                         (key absorption)
 *   s[b,h,t]     = scale * (q_lat[b,h,:] . c_t + q_pe[b,h,:] . k_pe_t)
 *   p            = softmax_t(s)           (split over the sequence, merged by LSE)
 *   o_lat[b,h,:] = sum_t p[b,h,t] c_t                               (latent sum)
 *   out[b,h,:]   = W_UV[h] o_lat[b,h,:]                              (value absorption)
 * Sources: "DeepSeek MLA 吸收式缓存：真实权重执行与 FlashMLA 架构边界"
 * (DEEPSEEK_MLA_ABSORB_AUDIT.md) §2.2 (q^T W_UK c = (W_UK^T q)^T c), §2.3
 * (sum_t p_t W_UV c_t = W_UV sum_t p_t c_t), §2.4 (the 64-wide RoPE key is
 * cached beside the 512-wide latent: 576 elements per token and layer), §6.1
 * (MQA mode over the latent: key width 576, value width 512); "手搓 MLA:从 MHA
 * 到 weight absorption" §四 (the absorbed einsums).  Cache quantization:
 * "DeepSeek-V2-Lite MLA 吸收式 KV 缓存优化 — 完整实验报告" §3.2 (per-channel
 * INT8 in 32-element blocks, asymmetric INT4 in 32-element blocks, k_pe INT8
 * in 8-element blocks).
 *
 * Conventions for every call below.
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    allocates and frees nothing.  bf16 means IEEE bfloat16 bit patterns.
 *  - Calls are asynchronous on `stream` and never synchronise the host, except
 *    mla_get_device_status.
 *  - Argument checks happen on the host before anything is enqueued; a failed
 *    check returns a negative mla_status_t and enqueues nothing.
 *  - Problems only the device can see (a page id outside the pool, a sequence
 *    longer than its page-table row, a bounded wait that gave up) are recorded
 *    in a device status word; the affected kernel skips the bad access (it
 *    substitutes page 0, or clamps the length) and the first such error is
 *    reported by mla_get_device_status.
 *  - The functions act on the CUDA device current on the calling thread.
 *  - The library resolves device addresses of its own globals (the status
 *    word, the no-allocation scratch) once per device and keeps them for the
 *    life of the process: do not use it across a device reset
 *    (cudaDeviceReset) or any other teardown of the device's primary context.
 *  - No C++ exception crosses this interface.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Fixed MLA dimensions (DeepSeek-V2-Lite and DeepSeek-V3 attention layers). */
#define MLA_D_C 512      /* kv_lora_rank: width of the cached latent c_KV      */
#define MLA_D_R 64       /* qk_rope_head_dim: width of the shared RoPE key     */
#define MLA_D_NOPE 128   /* qk_nope_head_dim                                  */
#define MLA_D_V 128      /* v_head_dim                                        */
#define MLA_PAGE 64      /* tokens per cache page                              */

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID = -1,      /* null pointer, negative size, misaligned buffer        */
  MLA_ERR_UNSUPPORTED = -2,  /* head count or format outside the supported set        */
  MLA_ERR_CUDA = -3,         /* a CUDA runtime call (launch, attribute) failed        */
  MLA_ERR_BOUNDS = -4,       /* device: page id outside the pool / sequence too long  */
  MLA_ERR_TIMEOUT = -5,      /* device: a bounded wait inside a kernel gave up        */
  MLA_ERR_WORKSPACE = -6     /* workspace smaller than mla_decode_workspace_bytes     */
} mla_status_t;

/* Cache storage formats. */
typedef enum {
  MLA_FMT_BF16 = 0,       /* c_KV and k_pe in bfloat16                                   */
  MLA_FMT_INT8 = 1,       /* c_KV INT8 per 32-channel group, k_pe INT8 per 8, bf16 scales */
  MLA_FMT_INT4 = 2,       /* c_KV asymmetric INT4 per 32 (bf16 scale + zero), k_pe INT8/8 */
  MLA_FMT_INT8_TOKEN = 3, /* c_KV INT8 with one scale per token, k_pe INT8/8 (INT8 pages) */
  MLA_FMT_INT4_SYM = 4,   /* c_KV symmetric INT4 per 32, k_pe INT8/8 (INT4 pages)         */
  MLA_FMT_INT4_PE4 = 5    /* c_KV asymmetric INT4 per 32, k_pe symmetric INT4/8 (INT4 pages) */
} mla_fmt_t;

/*
 * Page layout (one physical page = MLA_PAGE token slots; section offsets are
 * in bytes from the start of the page; per-slot rows are contiguous):
 *
 * MLA_FMT_BF16, 73,728 B:  [0)      slot s: 576 bf16 = c_KV[0..511], k_pe[0..63]
 * MLA_FMT_INT8, 39,936 B:  [0)      c codes    int8 [64][512]
 *                          [32768)  k_pe codes int8 [64][64]
 *                          [36864)  c scales   bf16 [64][16]   (group g = channels 32g..32g+31)
 *                          [38912)  k_pe scale bf16 [64][8]    (group g = dims 8g..8g+7)
 * MLA_FMT_INT4, 25,600 B:  [0)      c codes    u8   [64][256]  (channel 2i low nibble, 2i+1 high)
 *                          [16384)  k_pe codes int8 [64][64]
 *                          [20480)  c scales   bf16 [64][16]
 *                          [22528)  c zeros    bf16 [64][16]
 *                          [24576)  k_pe scale bf16 [64][8]
 * Quantizer (fp32 arithmetic, bit-exact and deterministic):
 *   INT8 group:  s = bf16_rne(amax / 127); code = clamp(rint(x / s), -127, 127); x^ = code * s
 *   INT4 group:  s = bf16_rne((max - min) / 15); z = min;
 *                code = clamp(rint((x - z) / s), 0, 15); x^ = code * s + z
 *   rint rounds half to even; a group with s == 0 stores zero codes.
 * The other quantizers "DeepSeek-V2-Lite MLA 吸收式 KV 缓存优化" §3.2 compares
 * write the same two page layouts, so the decode reads them unchanged:
 *   MLA_FMT_INT8_TOKEN (INT8 pages): s = bf16_rne(amax over the token's 512
 *     channels / 127), stored in all 16 of its c scale slots; codes as INT8.
 *   MLA_FMT_INT4_SYM (INT4 pages): per 32-channel group s = bf16_rne(amax / 7),
 *     q = clamp(rint(x / s), -7, 7) (0 when s == 0), stored as the nibble q + 8
 *     with zero = -8 s (exact in bf16), so that code * s + zero = q * s.
 *   MLA_FMT_INT4_PE4 (INT4 pages): c_KV as MLA_FMT_INT4; the RoPE key symmetric
 *     INT4 per 8-dim group ("k_pe 对称 INT4 (8块)"): s = bf16_rne(amax / 7),
 *     q = clamp(rint(x / s), -7, 7) (0 when s == 0), stored as INT8 codes in
 *     the page's k_pe code section with s in its k_pe scale slot, so x^ = q * s
 *     as for the INT8 RoPE key (4 bits of precision in an 8-bit slot: the
 *     quantizer's accuracy, not its smaller footprint).
 * (One scale for the whole tensor cannot serve an append-only cache: it would
 * change as tokens arrive.)
 */
typedef struct {
  int fmt;          /* mla_fmt_t                                                  */
  int num_pages;    /* physical pages in the pool                                 */
  void* pages;      /* device, num_pages * mla_cache_page_bytes(fmt) bytes,
                       256-byte aligned; owned by the caller                       */
} mla_cache_t;

/* Bytes of one physical page of `fmt` (0 for an unknown format). */
size_t mla_cache_page_bytes(int fmt);

/*
 * Split the up-projection wkv_b into the absorbed weights.
 *   wkv_b : bf16 [H*(128+128)][512]; rows h*256 .. h*256+127 are head h's
 *           no-RoPE key projection, the next 128 rows its value projection
 *           ("手搓 MLA" §三, k_nope, v = split(kv_up), read per head).
 *   W_UK  : bf16 [H][512][128], written; W_UK[h][c][d] = wkv_b[h*256 + d][c]
 *           (the key projection stored transposed, d fastest).
 *   W_UV  : bf16 [H][128][512], written; W_UV[h][d][c] = wkv_b[h*256 + 128 + d][c].
 * Bit-exact copy.  H in {16, 128}.  All three buffers 16-byte aligned.
 */
int mla_absorb_weights(const void* wkv_b, int H, void* W_UK, void* W_UV, cudaStream_t stream);

/*
 * Append T new tokens to each of B sequences.
 *   c_kv       : bf16 [B][T][512], k_pe : bf16 [B][T][64] (k_pe already RoPE-rotated)
 *   page_table : int32 [B][max_pages]; logical page j of row b lives in physical
 *                page page_table[b*max_pages + j]
 *   pos        : int32 [B] (device): token t of row b goes to position pos[b]+t,
 *                i.e. page (pos[b]+t)/64, slot (pos[b]+t)%64
 * The token's payload is written (quantized when cache->fmt asks for it);
 * nothing else in the pool changes.  A position beyond max_pages*64 or a
 * page id outside [0, num_pages) is skipped and raises MLA_ERR_BOUNDS.
 * Rows of the same call must not target the same slot.
 */
int mla_cache_append(const mla_cache_t* cache, const void* c_kv, const void* k_pe,
                     const int32_t* page_table, int max_pages, const int32_t* pos,
                     int B, int T, cudaStream_t stream);

/*
 * The step before the append, fused with it: computes each new token's cache
 * payload from its attention input and writes it like mla_cache_append.
 * "手搓 MLA" §三: c_kv = rmsnorm(x W_DKV^T, W_KVN), k_pe = rope(x W_KR^T);
 * "DeepSeek MLA 吸收式缓存" §3.3 names the joint projection wkv_a
 * (kv_a_proj_with_mqa) and the gain kv_norm.
 *   x          : bf16 [B][T][hidden], the attention inputs of the new tokens
 *   hidden     : a multiple of 64 in [64, 65536] (2048 for V2-Lite, 7168 for V3),
 *                else MLA_ERR_UNSUPPORTED
 *   wkv_a      : bf16 [576][hidden]; rows 0..511 are W_DKV (the latent), rows
 *                512..575 W_KR (the shared RoPE key)
 *   kv_norm_w  : bf16 [512], the RMSNorm gain W_KVN
 *   eps        : RMSNorm epsilon, >= 0 (1e-6 for these models)
 *   rope_theta : RoPE base, > 0 (10000 for these models)
 *   page_table, max_pages, pos, B, T : as for mla_cache_append; token t of row b
 *                has position pos[b]+t, which also sets its rotation
 *   latent_out : NULL, or bf16 [B][T][576]: receives each token's payload
 *                before quantization (c_kv then k_pe, the bf16 values a bf16
 *                pool would hold), whether or not its page write succeeded
 *   k_splits   : 0 picks the kernel and the split of the projection's K
 *                dimension by size (at most 64 tokens in all: a warp-level MMA
 *                kernel, one CTA per 64 output columns and hidden slice of at
 *                most 512); n > 0 forces the tcgen05 kernel with n CTA pairs
 *                per 128-token tile (capped at hidden/64; MLA_ERR_UNSUPPORTED if
 *                the tiles times the pairs exceed a grid)
 *   workspace  : device scratch of >= mla_cache_project_workspace_bytes(B, T,
 *                hidden, k_splits) bytes, 256-byte aligned (may be NULL when that
 *                is 0); every byte the call reads it writes first (the split
 *                pairs' partial payloads), so calls that share one workspace
 *                must not overlap on the GPU
 * Per token, in fp32 from bf16 operands: y = wkv_a x (tensor cores, fp32
 * accumulation); c = y[0..511] / sqrt(mean(y[0..511]^2) + eps) * kv_norm_w;
 * pairs (2i, 2i+1) of y[512..575] rotated by the angle pos * rope_theta^(-2i/64)
 * (reduced to one turn in 64-bit fixed point: the frequency as a fraction of
 * a turn in units of 2^-64, times pos modulo 2^64; angle error under 1e-6 rad
 * for any int32 position); each value rounded once to bf16,
 * then quantized exactly as mla_cache_append does.  With a K split each CTA's
 * partial product goes to its own slice of the workspace and a second kernel
 * (one CTA per token) sums the slices in split order before the same epilogue,
 * so the result is deterministic either way (the split count can change the
 * last bit of a value, being another fp32 summation order).  Bad
 * positions and page ids are skipped and raise MLA_ERR_BOUNDS as in
 * mla_cache_append.  x, wkv_a, kv_norm_w and latent_out 16-byte aligned.
 * Formats MLA_FMT_BF16, MLA_FMT_INT8 and MLA_FMT_INT4; the per-token INT8 and
 * symmetric INT4 variants return MLA_ERR_UNSUPPORTED here (append their
 * payload, from latent_out of a bf16 call, with mla_cache_append).
 */
int mla_cache_project_append(const mla_cache_t* cache, const void* x, int hidden, const void* wkv_a,
                             const void* kv_norm_w, float eps, float rope_theta,
                             const int32_t* page_table, int max_pages, const int32_t* pos,
                             int B, int T, void* latent_out, int k_splits,
                             void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Workspace for mla_cache_project_append on the current device (0 when no K
 * split is used, or for arguments that call would reject). */
size_t mla_cache_project_workspace_bytes(int B, int T, int hidden, int k_splits);

/*
 * Workspace needed by mla_decode for B rows and H heads on the current
 * device (the split-KV partials, the query-side latent and the split plan).
 */
size_t mla_decode_workspace_bytes(int B, int H);

/*
 * One absorbed decode step (q_len = 1 per row).
 *   q_nope    : bf16 [B][H][128]      q_pe : bf16 [B][H][64] (RoPE-rotated)
 *   W_UK      : bf16 [H][512][128]    W_UV : bf16 [H][128][512] (mla_absorb_weights)
 *   cache     : the page pool; page_table int32 [B][max_pages]
 *   seqlens   : int32 [B] (device): row b attends to its tokens 0 .. seqlens[b]-1
 *               (the new token included when it was appended first).  A row
 *               with seqlen 0 produces zeros.
 *   scale     : softmax scale, > 0 (1/sqrt(192) for these models)
 *   workspace : device scratch of >= mla_decode_workspace_bytes(B, H) bytes,
 *               256-byte aligned; contents need no initialisation
 *   out       : bf16 [B][H][128], written
 * H in {16, 128}: H = 128 runs the tcgen05 tensor-core kernel, H = 16 the
 * warp-level MMA kernel (or the CUDA-core kernel, mla_decode_select_kernel).
 * Formats: H = 128 reads bf16, INT8 and INT4 pools (codes
 * are dequantized to bf16 in the kernel's load stage, x = code*s (+ z), fp32
 * then one bf16 rounding); H = 16 reads bf16 pools only (MLA_ERR_UNSUPPORTED
 * otherwise).  Equivalent to mla_decode_plan + mla_decode_absorb_q +
 * mla_decode_attend + mla_decode_combine on the same stream.
 * The softmax is exact for every input ("DeepSeek MLA 吸收式缓存" §2.3 and the
 * online softmax it rests on): the H = 128 kernel tracks a lazily moved
 * reference maximum and exchanges half scores in fp16; a row whose scores
 * jump more than 2^100 above that reference, or whose half scores exceed 32
 * in magnitude (log2 units), is flagged by it and recomputed by
 * mla_decode_combine with an online softmax that rescales at every new
 * maximum (fp32, straight from the cache), so such rows cost more time, not
 * accuracy.
 */
int mla_decode(const void* q_nope, const void* q_pe, const void* W_UK, const void* W_UV, int H,
               const mla_cache_t* cache, const int32_t* page_table, int max_pages,
               const int32_t* seqlens, int B, float scale,
               void* workspace, size_t workspace_bytes, void* out, cudaStream_t stream);

/* The four steps of mla_decode, callable one by one (same arguments). */

/* Step 0: split plan.  Cuts the rows' 64-token pages into contiguous,
 * near-equal ranges, one per persistent worker of the attend kernel that
 * (H, fmt) selects; stored in the workspace.  Lengths beyond max_pages*64
 * are clamped and raise MLA_ERR_BOUNDS (negative lengths count as 0). */
int mla_decode_plan(int H, int fmt, const int32_t* seqlens, int B, int max_pages,
                    void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Step 0 with a chosen number of split workers, 1 <= workers <=
 * mla_decode_max_workers(H, fmt) (MLA_ERR_INVALID otherwise); the steps after
 * it follow the plan.  The split count changes only where the sequence is cut
 * into partials, so results agree with the default plan's within the stated
 * tolerance (not bit for bit).  For tests of that invariance and for
 * load-balance studies; mla_decode uses the default. */
int mla_decode_plan_workers(int H, int fmt, const int32_t* seqlens, int B, int max_pages, int workers,
                            void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* The default (largest) number of split workers of the attend kernel for H
 * heads over a `fmt` cache on the current device: persistent CTA pairs of the
 * tcgen05 kernel, CTAs of the 16-head kernels; a negative status for an
 * unsupported pair. */
int mla_decode_max_workers(int H, int fmt);

/* Step 1: q_lat = W_UK^T q_nope (fp32 accumulation, rounded to bf16) and
 * q_pe, stored in the workspace as the query operand of step 2.  Every input
 * is read after the kernel before this call in the stream has completed, so
 * that kernel may be the one that wrote W_UK (mla_absorb_weights). */
int mla_decode_absorb_q(const void* q_nope, const void* q_pe, const void* W_UK, int H, int B,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Step 2: the split-KV online-softmax pass over the plan of step 0; leaves
 * per-split (o_lat / l, LSE) partials in the workspace.  Reads the lengths
 * as clamped by step 0. */
int mla_decode_attend(int H, const mla_cache_t* cache, const int32_t* page_table, int max_pages,
                      const int32_t* seqlens, int B, float scale,
                      void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Step 3: LSE-merge of the splits into o_lat, then out = W_UV o_lat (bf16).
 * o_lat_out (fp32 [B][H][512]) may be NULL; when given, the merged latent
 * sum is stored there too.  W_UV is read as a weight: its first tiles load
 * while the kernel before this call in the stream (step 2) is still running,
 * so the kernel that wrote W_UV must not be the one directly before this
 * call.  Rows that step 2 flagged are recomputed here exactly from the cache
 * that step 2 read (its pointers are kept in the workspace), so the cache and
 * page table must be unchanged in between. */
int mla_decode_combine(const void* W_UV, int H, int B, void* workspace, size_t workspace_bytes,
                       void* out, float* o_lat_out, cudaStream_t stream);

/*
 * Several query tokens per row, causal: the absorbed attention of T new tokens
 * of every row over its cache (speculative / multi-token prediction decode, or
 * a prefill chunk run in absorbed form).  "手搓 MLA" §四 writes the absorbed
 * einsums with a query-token axis t (thd,hdc->thc; thc,sc->hts; hts,sc->thc;
 * thc,hdc->thd); "DeepSeek MLA 吸收式缓存" §3.4 runs the same layer as a
 * 25-token causal prefill and a 1-token incremental decode.
 *   q_nope    : bf16 [B][T][H][128]    q_pe : bf16 [B][T][H][64] (RoPE-rotated)
 *   seqlens   : int32 [B] (device): row b holds n_b >= T cached tokens whose
 *               last T are the queries (appended first): query t sits at
 *               position n_b - T + t and attends to tokens 0 .. n_b - T + t.
 *               n_b < T raises MLA_ERR_BOUNDS (queries then see no more than
 *               the row holds).
 *   workspace : >= mla_decode_q_workspace_bytes(B, H, T) bytes, 256-byte aligned
 *   out       : bf16 [B][T][H][128], written
 *   o_lat_out : NULL, or fp32 [B][T][H][512]: the merged latent sums
 * 1 <= T <= 65536, H in {16, 128}, every cache format; other arguments as
 * mla_decode.  Runs on the tcgen05 kernel for both head counts: its MMA has
 * 128 rows, so G = 128 / H query tokens of a row share one pass over the
 * row's cache (H = 16: 8 tokens, so the work per cached byte grows 8x;
 * H = 128: one token per pass) and each of those rows sees its own causal
 * prefix.  Same tolerance and exactness as mla_decode.
 */
int mla_decode_q(const void* q_nope, const void* q_pe, const void* W_UK, const void* W_UV, int H, int T,
                 const mla_cache_t* cache, const int32_t* page_table, int max_pages,
                 const int32_t* seqlens, int B, float scale,
                 void* workspace, size_t workspace_bytes, void* out, float* o_lat_out, cudaStream_t stream);

/* Workspace of mla_decode_q for B rows, H heads and T query tokens per row on
 * the current device (0 for arguments it would reject). */
size_t mla_decode_q_workspace_bytes(int B, int H, int T);

/*
 * The unabsorbed ("compute-friendly") causal prefill: the same attention as
 * mla_decode_q (T queries per row, the row's last T tokens, query t sees
 * tokens 0 .. n_b - T + t), computed by expanding every cached latent of the
 * rows into per-head keys and values once and running standard attention over
 * them.  "手搓 MLA" §三 (k_nope, v = split(kv_up); k = [k_nope; k_pe]) and its
 * closing notes (engines run this form at prefill, the absorbed one at decode);
 * "DeepSeek MLA 吸收式缓存" §2.1 (the expand path).  Per (query, key) pair it
 * costs 2H(192 + 128) FLOPs against the absorbed 2H(576 + 512), for a one-time
 * 2H x 256 x 512 per cached token.
 *   q_nope, q_pe, T, cache, page_table, max_pages, seqlens, B, scale, out : as mla_decode_q
 *   wkv_b     : bf16 [H*256][512], the joint up-projection (rows h*256.. : k_nope, then v)
 *   workspace : >= mla_prefill_workspace_bytes(B, H, max_pages) bytes, 256-byte
 *               aligned: the expanded keys and values, bf16 [B][max_pages*64][H][256]
 * bf16 pools only (MLA_ERR_UNSUPPORTED otherwise), H in {16, 128}.  Keys and
 * values are rounded to bf16 once after fp32 accumulation; the attention
 * accumulates in fp32.  Rows shorter than T raise MLA_ERR_BOUNDS.
 */
int mla_prefill(const void* q_nope, const void* q_pe, const void* wkv_b, int H, int T, const mla_cache_t* cache,
                const int32_t* page_table, int max_pages, const int32_t* seqlens, int B, float scale,
                void* workspace, size_t workspace_bytes, void* out, cudaStream_t stream);
size_t mla_prefill_workspace_bytes(int B, int H, int max_pages);

/*
 * The layer's output projection after the value up-projection:
 * y[r, :] = W_O . (out[r, 0, :], ..., out[r, H-1, :]), i.e. y = o Wo^T over
 * the heads' outputs side by side ("手搓 MLA" §三/§四 end both paths with
 * "@ Wo.T"; "DeepSeek MLA 吸收式缓存" §3.3 maps o_proj to wo).  It sums over
 * heads, so it follows the per-head merge as the next kernel of the chain:
 * called on the same stream right after mla_decode / mla_decode_q /
 * mla_prefill, it reads their bf16 output directly and streams its weight
 * while they finish (so the kernel that wrote W_O must not be the one
 * directly before this call in the stream).
 *   o         : bf16 [R][H][128] (the out of those calls; R = B, or B*T)
 *   W_O       : bf16 [hidden][H*128]
 *   hidden    : a multiple of 128, <= 65536 (2048 for V2-Lite, 7168 for V3)
 *   y         : bf16 [R][hidden], written (fp32 accumulation, one rounding)
 *   workspace : >= mla_output_projection_workspace_bytes(R, H, hidden) bytes,
 *               256-byte aligned (NULL when that is 0): fp32 sums when the
 *               reduction is split over several CTAs; cleared by the call, so
 *               calls sharing a workspace must not overlap on the GPU
 */
int mla_output_projection(const void* o, const void* W_O, int R, int H, int hidden, void* y,
                          void* workspace, size_t workspace_bytes, cudaStream_t stream);
size_t mla_output_projection_workspace_bytes(int R, int H, int hidden);

/*
 * Decode without any allocation (no counterpart on the pages: an interface
 * addition of this library for hosts that cannot allocate device memory, e.g.
 * an engine whose custom-op interface passes only inputs and outputs, a
 * runtime that owns all device memory through its own pool, or a serving loop
 * that forbids cudaMalloc once running).  Same arguments and result as
 * mla_decode, minus the workspace: the scratch is a fixed array of
 * MLA_NOALLOC_SCRATCH_BYTES in device global memory inside the library image,
 * held by every GPU that loads the library until the process exits.
 *  - All calls on a device share that array and it keeps the last call's
 *    contents; calls that overlap on the GPU race on it, so order them (one
 *    stream).  No part of it needs to start at zero.
 *  - The first call on a device resolves the array's address for that device
 *    (it must be current); make that first call before any stream capture.
 *  - A batch whose scratch cannot fit (even with a single split worker) is
 *    rejected with MLA_ERR_WORKSPACE; to fit, fewer split workers than
 *    mla_decode may be used, so results may differ in the last bits.
 *  - Calls no allocating routine.
 */
#define MLA_NOALLOC_SCRATCH_BYTES (64ull * 1024ull * 1024ull)
int mla_decode_noalloc(const void* q_nope, const void* q_pe, const void* W_UK, const void* W_UV, int H,
                       const mla_cache_t* cache, const int32_t* page_table, int max_pages,
                       const int32_t* seqlens, int B, float scale, void* out, cudaStream_t stream);

/*
 * Wait for `stream`, then return (and clear) the first device-detected error
 * recorded since the last call on the current device: MLA_OK, MLA_ERR_BOUNDS
 * or MLA_ERR_TIMEOUT (MLA_ERR_CUDA when the wait itself failed).  If `info` is
 * non-NULL it receives a detail value: the offending row or page id for
 * MLA_ERR_BOUNDS, the number of the wait site that gave up for MLA_ERR_TIMEOUT
 * (1 for mla_wait_selftest).
 */
int mla_get_device_status(cudaStream_t stream, int* info);

/*
 * Self-test of the device failure path.  Enqueues on `stream` one CTA pair
 * (a 2-CTA cluster, like the tcgen05 decode kernel) whose first CTA waits on a
 * barrier that nothing completes, through the same bounded wait the decode
 * kernel uses.  After that wait's limit (about 2 s at the maximum SM clock)
 * it gives up, records MLA_ERR_TIMEOUT with detail 1 in the device status
 * word and raises the abort flags of both CTAs; the second CTA, which starts
 * its own wait later, leaves it through the abort flag (as the other roles of
 * a decode kernel do).  The kernel then returns: nothing faults, the context
 * stays usable.  Read the outcome with mla_get_device_status.  Returns MLA_OK
 * once enqueued, MLA_ERR_CUDA if the launch fails.
 */
int mla_wait_selftest(cudaStream_t stream);

/* The split-KV attend kernels of the single-query decode.  H = 128 runs on the
 * fifth-generation tensor cores (tcgen05, a CTA pair per worker, every cache
 * format).  H = 16 over bf16 pages has two: the warp-level MMA kernel
 * (mma.sync m16n8k16, whose 16 rows are exactly the 16 heads; the default) and
 * the CUDA-core kernel (fp32 FMA; kept as the baseline the other is measured
 * against).  Both compute the defined softmax (fp32 online softmax with a
 * rescale at every new maximum). */
typedef enum {
  MLA_KERNEL_CUDA_CORES = 0,
  MLA_KERNEL_TCGEN05 = 1,
  MLA_KERNEL_MMA = 2
} mla_kernel_t;

/* Which attend kernel mla_decode (and the calls of its steps, and
 * mla_decode_noalloc) uses for H heads over bf16 pages: an mla_kernel_t value,
 * or -1 when H is unsupported. */
int mla_decode_kernel_kind(int H);

/* Selects the attend kernel for H heads, process-wide, for the calls that
 * start after it returns: H = 16 takes MLA_KERNEL_MMA or MLA_KERNEL_CUDA_CORES,
 * H = 128 only MLA_KERNEL_TCGEN05.  Returns MLA_OK or MLA_ERR_UNSUPPORTED.
 * The plan, attend and combine of one decode must see the same selection (do
 * not switch between mla_decode_plan and mla_decode_attend); the workspace
 * size does not depend on it. */
int mla_decode_select_kernel(int H, int kind);

/* Human-readable name of a status code (static string). */
const char* mla_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
