/*
 * lms.h -- C ABI of the GB300 (sm_103a) library for exact categorical token sampling fused
 * into the decode-time LM-head projection, with a Gumbel race over materialised logits and a
 * counter-based Philox noise generator.
 *
 * What the operations compute (sources are web pages, cited by title and section):
 *
 *  - "FlashSampling: fast and memory-efficient exact sampling" (summary of arXiv 2603.15854),
 *    "Gumbel-Max trick": i* = argmax_i (e_i + g_i) with g ~ Gumbel(0,1) is an exact sample of
 *    softmax(e).  "method step details": Stage 1 computes, per vocabulary tile, the logits
 *    Y = H W^T on chip (step 1), applies the deterministic transform (step 2), adds
 *    g = -log(-log u) (steps 3-4), keeps one (max, global index) candidate per row (step 5) and
 *    writes it to memory (step 6); Stage 2 takes, per row, the candidate of the best tile.
 *  - "Megatron-LM pull request 8370: fp64_sampling_noise", "Problem" and "The change": noise
 *    keyed by (request seed, absolute position, vocabulary index); float32 noise loses the tail
 *    beyond ~20 nats; two Philox words give a 52-bit midpoint uniform (k + 1/2)/2^52 that keeps
 *    it to ~40 nats.  The same page ("Cost") proposes generating the noise in registers with
 *    several blocks per row over materialised logits: lms_sample_from_logits.
 *  - "Write Triton Sampling Kernel", reasoning steps 3-4 and "Kernel design rules": bias is added
 *    before division by T; T == 0 short-circuits to argmax; ties go to the smallest index;
 *    masked / out-of-range entries are -inf.
 *
 * Exact definitions used by every entry point (identical on all paths):
 *   Philox       Philox4x32, 10 rounds (Salmon et al., SC'11): call(key, counter) -> words
 *                w0..w3.  key = (k0, k1), counter = (c0, c1, c2, c3), all 32-bit.
 *   key/counter  seeded row b (seeds[b] >= 0): key = (seed lo32, seed hi32), and call n has
 *                counter (n, pos lo32, pos hi32, 0) with pos = positions[b]; unseeded row b:
 *                key = (base_seed lo32, base_seed hi32), and call n has counter
 *                (n, offset lo32, offset hi32, 0x80000000 | b), b the row's index in the call.
 *   entry words  one call serves several consecutive vocabulary entries, and no word is
 *                dropped.  FP32 noise: entry v takes word w[v & 3] of call n = v >> 2.
 *                WIDE53 noise: entry v takes lo = w[2 (v & 1)] and hi = w[2 (v & 1) + 1] of
 *                call n = v >> 1.  The variate of entry v is thus a function of (key, counter
 *                words 1..3, v) alone: a seeded row's noise depends on (seed, position, v), not
 *                on the row's place in the batch.
 *   uniform      FP32 noise: k = w >> 8 (w the entry's word), u = (k + 1/2) / 2^24 = (2k + 1) / 2^25.
 *                WIDE53 noise: k = ((hi << 32) | lo) >> 12, u = (k + 1/2) / 2^52 = (2k + 1) / 2^53.
 *   noise        E = -log u, g = -log E (computed in fp32 from exact integer-derived u or 1 - u).
 *   transform    masked -> -inf; T == 0 -> s = y + bias (greedy, no noise);
 *                T > 0 -> s = (y + bias) / T + g;  NaN scores count as -inf.
 *   race         per row, the largest s; ties -> smallest v; -inf never wins.
 *   row status   0 ok; 1 no entry above -inf (index -1); 2 T < 0 or NaN (index -1);
 *                3 a device-side wait ran out of time (index -1; the call's results for that
 *                row are void, the CUDA context stays usable).
 *
 * Conventions: all data pointers are DEVICE memory owned by the caller; the library never
 * allocates, frees or retains them.  Calls are asynchronous on `stream` (a cudaStream_t; NULL =
 * the legacy default stream).  Host-detectable errors return a non-zero lms_status before
 * anything is launched; lms_last_error() then holds a message (thread-local).  Between calls the
 * library keeps only per-device launch settings (kernel attributes and occupancy checks, set once
 * under a lock) and, for lms_lmhead_sample_noalloc, its static scratch; no call's data outlives it.
 */
#ifndef LMS_H_
#define LMS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LMS_OK = 0,
    LMS_ERR_INVALID_ARG = 1,  /* null required pointer, size <= 0 or too large, bad enum value */
    LMS_ERR_UNSUPPORTED = 2,  /* alignment / shape the kernels do not handle (see each call)    */
    LMS_ERR_WORKSPACE = 3,    /* workspace NULL or smaller than lms_workspace_bytes()           */
    LMS_ERR_CUDA = 4,         /* a CUDA runtime / driver call failed (message in last_error)   */
    LMS_ERR_TIMEOUT = 5       /* lms_read_status only: a device-side wait of the call ran out
                                 of time (some row ended with status 3)                       */
} lms_status;

typedef enum { LMS_NOISE_FP32 = 0, LMS_NOISE_WIDE53 = 1 } lms_noise_mode;
typedef enum { LMS_DTYPE_F32 = 0, LMS_DTYPE_BF16 = 1 } lms_dtype;
typedef enum {
    LMS_NOISE_OUT_WORDS = 0,      /* uint32 [B][V][4]: the four words of the Philox call entry v
                                     draws from (entries served by one call repeat them)       */
    LMS_NOISE_OUT_UNIFORM = 1,    /* double [B][V]: u, exact                                    */
    LMS_NOISE_OUT_EXPONENTIAL = 2,/* float  [B][V]: E = -log u as the sampling kernels compute it */
    LMS_NOISE_OUT_GUMBEL = 3      /* float  [B][V]: g = -log E as the sampling kernels compute it */
} lms_noise_kind;
typedef enum { LMS_OP_LMHEAD = 0, LMS_OP_LOGITS = 1, LMS_OP_LMHEAD_FP8 = 2 } lms_op;
typedef enum {
    LMS_PATH_AUTO = 0,            /* the library's choice (currently tcgen05 for every B)      */
    LMS_PATH_GEMV = 1,            /* CUDA-core dot products (B <= LMS_GEMV_MAX_B)                */
    LMS_PATH_TCGEN05 = 2,         /* TMA -> shared memory -> tcgen05.mma -> TMEM accumulators  */
    LMS_PATH_TCGEN05_PAIR = 3     /* the same on CTA pairs: tcgen05.mma.cta_group::2, M = 256;
                                     each CTA streams half of H (for large batches)            */
} lms_path;

#define LMS_ROW_OK 0
#define LMS_ROW_NO_CANDIDATE 1
#define LMS_ROW_BAD_TEMPERATURE 2
#define LMS_ROW_DEVICE_TIMEOUT 3

#define LMS_GEMV_MAX_B 8
#define LMS_FUSED_TILE_V 128

/* Fault injection for tests of the timeout path only (0 in normal use): the fused tcgen05
 * kernel's first CTA never issues its first shared-memory load, so the wait on it runs out. */
#define LMS_DEBUG_WITHHOLD_FIRST_LOAD 1u

typedef struct {
    const float* temperature;   /* [B] or NULL (all 1).  0 = greedy row; < 0 or NaN = status 2 */
    const int64_t* seeds;       /* [B] or NULL (all unseeded).  seeds[b] < 0 = unseeded row    */
    const int64_t* positions;   /* [B] absolute position of the token being drawn; read for
                                   seeded rows (required when seeds != NULL)                 */
    const float* bias;          /* [B][ld_bias] fp32 additive bias or NULL; ld_bias == 0 shares
                                   one [V] row across the batch.  May hold -inf.             */
    int64_t ld_bias;
    const uint32_t* allow_mask; /* [B][ld_mask] words or NULL: bit (v % 32) of word (v / 32)
                                   set = token v allowed.  ld_mask == 0 shares one row.      */
    int64_t ld_mask;
    uint64_t base_seed;         /* key of unseeded rows                                       */
    uint64_t offset;            /* step counter of unseeded rows; advance it every step      */
    int32_t noise_mode;         /* lms_noise_mode                                             */
    int32_t tile_v;             /* 0 = automatic; see lms_tile_info for the allowed values    */
    int32_t path;               /* lms_path (fused entry point only)                          */
    uint32_t timeout_ms;        /* bound on each device-side wait; 0 = 2000 ms                */
    int32_t* row_status;        /* [B] per-row status out, or NULL                            */
    uint32_t debug_flags;       /* 0, or LMS_DEBUG_* for fault-injection tests                */
    uint32_t reserved;          /* must be 0                                                  */
} lms_sample_params;

/* Library version string. */
const char* lms_version(void);

/* Message for the last non-OK return on this thread ("" if none). */
const char* lms_last_error(void);

/* Tiling the entry point `op` will use for a call of these sizes.  tile_v_req = 0 asks for the
 * automatic choice.  LMS_OP_LMHEAD: tile_v is 128 (one tcgen05 M=128 tile per vocabulary tile;
 * the GEMV path uses the same tiles).  LMS_OP_LOGITS: tile_v is a power of two in
 * [256, 65536].  Outputs (any may be NULL): the tile width, the number of vocabulary tiles
 * nt = ceil(V / tile_v), the workspace size in bytes, and (fused op) the path auto selects.
 * D is ignored for LMS_OP_LOGITS. */
lms_status lms_tile_info(int32_t op, int64_t B, int64_t D, int64_t V, int32_t tile_v_req,
                         int32_t* tile_v_out, int64_t* n_tiles_out, size_t* workspace_bytes_out,
                         int32_t* path_out);

/* Workspace bytes for a call of these sizes (0 if the sizes are invalid).  Every workspace (of
 * every entry point that takes one) starts with a 256-byte status block: uint32 status word at
 * offset 0 (see lms_read_status), the rest reserved.  Then, for LMS_OP_LMHEAD and LMS_OP_LOGITS,
 * for tests that read the Stage-1 candidates: float score[B][nt] at offset 256, then int32
 * index[B][nt] at offset 256 + round_up(4*B*nt, 256).  index -1 = tile had no entry above -inf.
 * Nothing in a workspace has to be initialised by the caller. */
size_t lms_workspace_bytes(int32_t op, int64_t B, int64_t D, int64_t V, int32_t tile_v_req);

/* The status of the last call that used `workspace` (any entry point that takes a workspace),
 * for callers that pass row_status = NULL.  Synchronises `stream` (the call's stream), then reads
 * the status word that the call left at the head of the workspace: bit s is set when at least
 * one row ended with row status s (1 no finite score, 2 invalid T, 3 a device-side wait ran out);
 * 0 when every row is OK.  *status_bits receives the word (status_bits may be NULL).  Returns
 * LMS_ERR_TIMEOUT when bit 3 is set, LMS_OK otherwise (LMS_ERR_CUDA if the synchronisation or
 * the 4-byte copy fails).  Allocates nothing.  (FlashSampling "Limitations": the kernel assumes
 * at least one finite logit per row; status 1 reports a row without one, and this call lets a
 * caller without a row_status buffer see it.) */
lms_status lms_read_status(const void* workspace, void* stream, uint32_t* status_bits);

/* Fused LM-head projection + Gumbel-max sampling (FlashSampling Stage 1 + Stage 2).
 *   H   bf16 [B][ldh] hidden states (row-major), W bf16 [V][ldw] LM-head weight (row-major, the
 *       vocabulary-major layout the FlashSampling page uses for W in R^{V x D}).
 *   out int64 [B]: the sampled token per row (-1 when row status != 0).
 * Logits are never written to memory: each CTA keeps its [128 x B] tile on chip (TMEM or
 * registers) and writes one (score, index) candidate per row to the workspace; Stage 2 reduces
 * them.  Requirements (LMS_ERR_UNSUPPORTED otherwise): D % 8 == 0, ldh and ldw multiples of
 * 8 elements, H and W 16-byte aligned, 1 <= B <= 65536, 1 <= V < 2^31, D <= 65536.
 * LMS_PATH_GEMV needs B <= LMS_GEMV_MAX_B. */
lms_status lms_lmhead_sample(const void* H, int64_t ldh, const void* W, int64_t ldw, int64_t B,
                             int64_t D, int64_t V, const lms_sample_params* params, int64_t* out,
                             void* workspace, size_t workspace_bytes, void* stream);

/* The fused path with FP8 (E4M3) inputs, W8A8 (FlashSampling "Limitations": low-precision FP8
 * inputs, which the kernel structure supports):
 *   W8      E4M3 [V][ldw8] bytes ("fn" encoding: no infinities, max 448), w_scale fp32 [V]: the
 *           weight is W[v][d] = E4M3(W8[v][d]) * w_scale[v] (quantised by the caller, offline).
 *   H       bf16 [B][ldh], quantised by the call: row b is scaled by 2^-e_b, e_b the smallest
 *           integer with max_d |H[b][d]| * 2^-e_b <= 448, and rounded to the nearest E4M3 value
 *           (ties to even).  The power-of-two scale makes the scaling exact.
 * Logits y[b][v] = 2^e_b * w_scale[v] * sum_d E4M3(H8[b][d]) E4M3(W8[v][d]) (tcgen05.mma
 * kind::f8f6f4, fp32 accumulation); everything after that is lms_lmhead_sample's.  W streams at
 * one byte per weight.  Workspace (lms_workspace_bytes(LMS_OP_LMHEAD_FP8, ...)): the status block
 * and the candidates as for lms_lmhead_sample, then the quantised activations [B][round_up(D, 16)]
 * bytes, then e_b int32 [B], each at a 256-byte aligned offset.  Requirements: D % 16 == 0, ldw8 >= D and % 16 == 0, ldh as for
 * lms_lmhead_sample, H and W8 16-byte aligned; path AUTO or TCGEN05. */
lms_status lms_lmhead_sample_fp8(const void* H, int64_t ldh, const void* W8, int64_t ldw8,
                                 const float* w_scale, int64_t B, int64_t D, int64_t V,
                                 const lms_sample_params* params, int64_t* out, void* workspace,
                                 size_t workspace_bytes, void* stream);

/* The fused path with MXFP4 weights and bf16 activations (W4A16; FlashSampling "Limitations" and
 * "Future directions": low-precision inputs for the memory-bound regime).  The weight format is
 * the Open Compute Project's Microscaling MXFP4.  Its logical layout, which lms_mxfp4_pack reads:
 *   W4   uint8 [V][ldw4] (ldw4 >= D/2): element d of row v is the low nibble of byte d/2 when d
 *        is even, the high nibble when odd; an E2M1 code (bit 3 sign, bits 2..1 exponent with
 *        bias 1, bit 0 mantissa: 0, 0.5, 1, 1.5, 2, 3, 4, 6 and negatives).
 *   S    uint8 [D/32][lds] (lds >= V), block-major: S[k][v] is the UE8M0 scale code of elements
 *        32k..32k+31 of row v; the scale is 2^(S - 127).
 *   W[v][d] = E2M1(code) * 2^(S[d/32][v] - 127).
 * lms_mxfp4_pack rewrites a matrix once into the library's tiled device format (Wt,
 * lms_mxfp4_tiled_bytes(V, D) bytes): one contiguous 4352-byte block per 128-row vocabulary tile
 * and 64-element K chunk (4 KB of codes, row r at byte 32 r; then the two blocks' 128 scale codes
 * each), so that each block streams with a single contiguous copy.  A row's 32 code bytes are
 * eight little-endian 32-bit words of eight consecutive elements e0..e7: the magnitude bits
 * (bits 2..0 of the code) of e_k at bits 4k..4k+2, the sign of e_k at bit 8k+7 for k < 4 and at
 * bit 8(k-4)+3 for k >= 4, which lets the sign join its bf16 high byte with one logic operation.
 * Rows past V and elements past D are zero.  lms_lmhead_sample_mxfp4 then computes logits y[b][v] = sum_d H[b][d] W[v][d] with
 * fp32 accumulation; everything after that is lms_lmhead_sample's (same noise, transform, race,
 * statuses and workspace: lms_workspace_bytes(LMS_OP_LMHEAD, ...)).  The weights stream at 0.53
 * bytes each and are rebuilt on chip as exact bf16 values; that is exact for scale codes 3..252
 * (2^-124 .. 2^125), the range any real weight matrix quantises to.
 * Requirements: D % 32 == 0, D <= 65536; lms_lmhead_sample_mxfp4: ldh as for lms_lmhead_sample,
 * H and Wt 16-byte aligned, Wt_bytes >= lms_mxfp4_tiled_bytes(V, D), path AUTO or TCGEN05. */
size_t lms_mxfp4_tiled_bytes(int64_t V, int64_t D);
lms_status lms_mxfp4_pack(const void* W4, int64_t ldw4, const void* S, int64_t lds, int64_t V, int64_t D,
                          void* Wt, size_t Wt_bytes, void* stream);
lms_status lms_lmhead_sample_mxfp4(const void* H, int64_t ldh, const void* Wt, size_t Wt_bytes, int64_t B,
                                   int64_t D, int64_t V, const lms_sample_params* params, int64_t* out,
                                   void* workspace, size_t workspace_bytes, void* stream);

/* Gumbel-top-k of the fused path: k draws without replacement per row (FlashSampling
 * "Limitations" and "Future directions": sampling without replacement by Gumbel-top-k, useful for
 * beam search).  The perturbed scores s = (y + bias) / T + g are lms_lmhead_sample's, with the
 * same noise; the call returns each row's k largest, larger score first, then the smaller index.
 * out[b][0] is the token lms_lmhead_sample draws.  Greedy rows (T == 0) get the k largest
 * y + bias.  Masked entries are never drawn.
 *   k        1 <= k <= LMS_TOPK_MAX
 *   out      int64 [B][k] (device): vocabulary indices; -1 past a row's finite scores
 *   scores   fp32 [B][k] (device) or NULL: the perturbed scores (-inf where out is -1)
 *   workspace  lms_workspace_bytes_topk(B, V, k) bytes: the 256-byte status block; ordered key
 *              lists in a region of uint64 [B][ceil(V / 128)][4][k]: one per row, tile and
 *              quarter of the tile's 128 rows ([B][ceil(V / 128)][4][k]), or, when
 *              4 * n_pad * k * 8 <= 32 KB (n_pad: min(B, 256) rounded up to a multiple of 16),
 *              one per row, Stage-1 CTA and quarter, each the k best keys of those rows over the
 *              CTA's tiles ([B][4 G][k], G = min(ceil(V / 128), SM count)); then, at the next
 *              256-byte boundary, Stage 2's per-row part lists uint64 [B][32][k] (written only when
 *              a row has more than 1024 lists and is split over several Stage-2 CTAs)
 * Row statuses as for lms_lmhead_sample (1: no finite score, 2: invalid T, 3: a bounded wait ran
 * out).  Requirements as for lms_lmhead_sample; path AUTO or TCGEN05 (bf16 H and W). */
#define LMS_TOPK_MAX 16
size_t lms_workspace_bytes_topk(int64_t B, int64_t V, int32_t k);
lms_status lms_lmhead_sample_topk(const void* H, int64_t ldh, const void* W, int64_t ldw, int64_t B,
                                  int64_t D, int64_t V, int32_t k, const lms_sample_params* params,
                                  int64_t* out, float* scores, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* Speculative-decoding verification (spec-decode-ops "verify": the canonical rejection sampling
 * of speculative decoding) over materialised logits.  For batch row b with draft tokens
 * x_0..x_{k-1} and p = softmax(logits / T) per position (T per row, for target and draft alike):
 * x_i is accepted when u_i * p_d(x_i) < p_t(x_i), i.e. with probability min(1, p_t / p_d), in
 * order; the first rejection j is replaced by a draw from the residual max(p_t - p_d, 0)
 * renormalised (the target's own draw if no entry of it is positive); with every draft
 * accepted, a bonus token is drawn from the target at position k.  The emitted tokens follow the
 * target's distribution exactly.  T == 0 rows accept while x_i is the target's argmax (smallest
 * index on ties) and then emit the argmax.  A draft token outside [0, V) is rejected.
 *   target   [B][k + 1] rows, draft [B][k] rows, each row ld >= V elements apart (fp32 or bf16)
 *   draft_tokens int64 [B][k]
 *   accept_len   int64 [B]: the accepted draft tokens j
 *   out          int64 [B][k + 1]: x_0..x_{j-1}, then the drawn token, then -1
 * Noise: the race's Philox noise for row b at absolute position positions[b] + i (seeded rows)
 * or row index b (k + 1) + i under (base_seed, offset) (unseeded rows); u_i is the same key's
 * call with counter word 0 = 0xffffffff (fp32 noise: its first word, wide noise: its first two).
 * params: temperature, seeds, positions, base_seed, offset, noise_mode, row_status (1: nothing
 * finite at the drawn position, 2: invalid T); bias, mask, tile_v, path and debug_flags must be
 * 0 / NULL.  1 <= k <= 32, V < 2^31.  Workspace: lms_workspace_bytes_verify(B, k, V). */
size_t lms_workspace_bytes_verify(int64_t B, int32_t k, int64_t V);
lms_status lms_verify_from_logits(const void* target, const void* draft, int32_t dtype, int64_t ld,
                                  int64_t B, int32_t k, int64_t V, const int64_t* draft_tokens,
                                  const lms_sample_params* params, int64_t* accept_len, int64_t* out,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* The same race over materialised logits [B][ld] (fp32 or bf16).  ld == 0 broadcasts one
 * row to all B draws (each draw keyed by its own row index / position).  Several CTAs share a
 * row (one per tile of tile_v entries); the noise is generated in registers.
 * Requirements: 1 <= B < 2^31, 1 <= V < 2^31; any alignment (16-byte aligned rows are read
 * with 128-bit loads). */
lms_status lms_sample_from_logits(const void* logits, int32_t dtype, int64_t ld, int64_t B,
                                  int64_t V, const lms_sample_params* params, int64_t* out,
                                  void* workspace, size_t workspace_bytes, void* stream);

/* Per-row filters for lms_sample_from_logits_filtered (all device arrays [B], each may be NULL).
 * spec-decode-ops "Semantics" and the sampling-kernel guide, reasoning steps 6-8:
 *   top_k  keep the k largest t = (y + bias) / T (ties: smaller index first).  Off when
 *          top_k[b] <= 0 or >= V; values above k_max count as k_max.
 *   top_p  keep the shortest prefix of that sorted set (or, with top-k off, of the first k_max
 *          tokens) whose probability mass, normalised over the set, reaches top_p; the crossing
 *          token is kept.  Off unless 0 < top_p[b] < 1.
 *   min_p  keep p >= min_p * p_max, i.e. t - t_max >= log(min_p).  Off unless 0 < min_p[b] <= 1.
 * Applied in this order; each keeps the top token.  The Gumbel race then runs over the kept
 * tokens with the same noise as lms_sample_from_logits, which samples the softmax renormalised
 * to them.  Greedy rows (T == 0) take the argmax. */
typedef struct {
    const int32_t* top_k;
    const float* top_p;
    const float* min_p;
    int32_t k_max;              /* candidate bound for top-k / top-p, 1..1024; 0 = 1024 */
    int32_t reserved;           /* must be 0 */
} lms_filter_params;

/* The filtered race over materialised logits [B][ld] (fp32 or bf16; ld == 0 broadcasts one row).
 * One thread-block cluster per row (up to 16 CTAs of 512 threads; CTA c owns one contiguous
 * slice of the row): each CTA keys its slice's t = (y + bias) / T in shared memory, the cluster
 * finds the top-k boundary by a radix select over histograms merged through distributed shared
 * memory, every CTA appends its surviving entries to the leader CTA, and the leader cuts top-p
 * (a radix select over exact fixed-point masses) and min-p (a threshold) and races what is left.
 * Nothing is sorted.  The leader's candidate list holds at most 2048 entries: the k_max best, or
 * the entries above the bin of the k-th one plus that whole bin when it holds at most 256 (ties
 * at the k-th value are then ranked among themselves).  out int64 [B] (-1 when row status != 0);
 * statuses through params->row_status only (no workspace).
 * Requirements: 1 <= B < 2^31, 1 <= V < 2^31. */
lms_status lms_sample_from_logits_filtered(const void* logits, int32_t dtype, int64_t ld, int64_t B,
                                           int64_t V, const lms_sample_params* params,
                                           const lms_filter_params* filters, int64_t* out,
                                           void* stream);

/* Allocation-free variant of lms_lmhead_sample for callers that cannot allocate device memory:
 * code that runs inside a device-memory allocator or a pool's callback, code that must not take
 * the allocator's lock, or an embedding that hands this library only fixed buffers.  The pages
 * have no counterpart of this call; it changes where the scratch lives, not what is computed.
 * Arguments and results are those of lms_lmhead_sample without the workspace: the Stage-1
 * candidates go to a 4 MiB file-scope device array that is part of the library image (every
 * GPU that loads the library holds it until the process exits), so B * ceil(V / 128) must be
 * <= 524288; larger calls return LMS_ERR_WORKSPACE before any launch.  Calls no cudaMalloc,
 * cudaFree or allocating library routine.  Each call made outside stream capture looks up the
 * array's device address (cudaGetSymbolAddress, with the call's device current), so a module
 * reloaded at a new address after cudaDeviceReset or in another context is picked up; calls made
 * while `stream` is capturing use the address the last uncaptured call on that device found, so
 * make a first call on each device (and again after a device reset or a context switch) before
 * any stream capture -- a captured first call returns LMS_ERR_CUDA.  Every call shares the array
 * and leaves its candidates in it; nothing in it has to start at zero (each call writes every
 * candidate it reads), but calls whose kernels overlap on the GPU (concurrent streams or threads)
 * race on it: serialise them.  Row statuses come through params->row_status only. */
lms_status lms_lmhead_sample_noalloc(const void* H, int64_t ldh, const void* W, int64_t ldw,
                                     int64_t B, int64_t D, int64_t V,
                                     const lms_sample_params* params, int64_t* out, void* stream);

/* Noise grid [B][V] as the sampling kernels compute it, for testing and debugging
 * (Megatron-LM PR 8370, "Tests": the noise replays bit-exactly; the words are the bit-exact
 * surface).  kind selects the output (lms_noise_kind; element sizes 16, 8, 4, 4 bytes);
 * noise_mode picks FP32 or WIDE53.  seeds / positions as in lms_sample_params. */
lms_status lms_philox_fill_noise(void* out, int32_t kind, int32_t noise_mode, int64_t B,
                                 int64_t V, const int64_t* seeds, const int64_t* positions,
                                 uint64_t base_seed, uint64_t offset, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* LMS_H_ */
