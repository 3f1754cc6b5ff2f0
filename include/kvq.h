/*
 * kvq.h -- C ABI of libkvq: single-token decode attention over a paged,
 * quantized KV cache, with the WitCert runtime error meter fused into the
 * attention pass.
 *
 * Sources (cited by page title and section):
 *   [W]  "WitCert: Sound Runtime Risk Observability and Gating for KV-Cache
 *        Quantization" (arXiv 2607.28699).
 *   [C]  "Compress the shared cartridge. Keep the keys." (knlp.io, cartridge
 *        asymmetric quantization).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Memory: the caller owns every buffer.  Pointers named *_dev are device
 *   pointers; the library never allocates, frees or resizes memory.
 * - Streams: work is enqueued on `stream` (a cudaStream_t; NULL is the legacy
 *   default stream) and the call returns without synchronising.  No entry
 *   point performs a host<->device copy or a host synchronisation, so the
 *   sequence append -> decode -> meter can be captured in a CUDA graph.
 * - Errors: argument errors are detected on the host and returned at once
 *   (nothing is enqueued).  Errors that only the device can see (a block-table
 *   entry or slot outside the cache, a non-finite input, a scale out of range,
 *   an asynchronous copy that never completed) are written to the caller's
 *   `err_word_dev` (a device int32 the caller zeroes) as the first kvq_status
 *   code observed (atomic compare-and-swap from 0); the kernels never trap and
 *   never spin without a bound.  Read it after synchronising the stream.
 * - Shapes: head_dim is 128, page size 16 tokens, 16 witness bands, at most 8
 *   query heads per kv head (GQA group G = num_q_heads / num_kv_heads <= 8).
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVQ_HEAD_DIM 128
#define KVQ_PAGE_SIZE 16
#define KVQ_N_BANDS 16
#define KVQ_MAX_GROUP 8
/* Largest num_kv_heads and batch kvq_decode_attn accepts (larger values: KVQ_ERR_INVALID_ARG). */
#define KVQ_MAX_KV_HEADS 128
#define KVQ_MAX_BATCH 1024
#define KVQ_VERSION 1

/* A cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st* kvq_stream_t;

typedef enum kvq_status {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1,         /* bad pointer, size, alignment or shape (host-detected)          */
  KVQ_ERR_UNSUPPORTED_LAYOUT = 2,  /* format / GQA group combination this build does not provide     */
  KVQ_ERR_WORKSPACE_TOO_SMALL = 3, /* ws_bytes < kvq_decode_workspace_size(...)                       */
  KVQ_ERR_CUDA = 4,                /* a CUDA runtime call or kernel launch failed                      */
  KVQ_ERR_DEVICE_BOUNDS = 5,       /* device: slot / block-table entry outside [0, num_pages*16)       */
  KVQ_ERR_NONFINITE_INPUT = 6,     /* device: non-finite key/value, or a scale that overflows fp16     */
  KVQ_ERR_RANGE = 7,               /* device: a value scale above KVQ_MAX_VALUE_SCALE (see kvq_append) */
  KVQ_ERR_TIMEOUT = 8              /* device: a bounded wait for an asynchronous copy gave up          */
} kvq_status;

/* Storage formats of one plane ([C] table "Keys carry the cartridge quantization loss"; [W] Sec. 4.2). */
typedef enum kvq_fmt {
  KVQ_FMT_BF16 = 0,        /* bfloat16, round-to-nearest-even; no scale                                  */
  KVQ_FMT_E4M3 = 1,        /* FP8 E4M3 raw cast, round-to-nearest-even, saturating at +-448; no scale     */
  KVQ_FMT_E4M3_SCALED = 2, /* FP8 E4M3 of x / s, s = fp16(amax / 448) per (token, kv head)               */
  KVQ_FMT_INT8_DITHER = 3, /* subtractively dithered INT8: code = rint(x/s + xi), s = fp16(amax / 126.5) */
  KVQ_FMT_INT8_DITHER_G32 = 4 /* the same with one scale per token per group of 32 channels: channels
                                 32g..32g+31 use s_g = fp16(amax_g / 126.5) ([W] Sec. 6.2.3, Table 4,
                                 G_c = 32); keys and values of one cache both in this format, no prefix,
                                 no key outlier bypass */
} kvq_fmt;

/* Element type of the key / value / query inputs. */
typedef enum kvq_dtype { KVQ_DTYPE_F32 = 0, KVQ_DTYPE_BF16 = 1 } kvq_dtype;

/* Largest per-token value scale the decode kernel accepts (the fp16 P*s*2^8 operand stays finite). */
#define KVQ_MAX_VALUE_SCALE 255.875f

/*
 * One layer's paged cache: planes of tiles, one tile per (page, kv head).
 * Tile index of (page p, kv head h) is p * num_kv_heads + h in the K, V and
 * witness planes and h * num_pages + p in the two scale planes and the value
 * witness plane (head-major, so that the small tiles of consecutive pages of
 * one head share a 128-byte memory line); a tile holds the 16 tokens (slots
 * p*16 .. p*16+15) of that page.  All planes are device memory, 16-byte
 * aligned, owned by the caller.
 *
 * Tile layouts (byte offset of token t in 0..15, channel c in 0..127, band b
 * in 0..15; they place each lane's tensor-core fragment in contiguous 16-byte
 * words so one bulk copy of a tile feeds the decode kernel with conflict-free
 * shared-memory loads):
 *   K, 16-bit (4096 B):  16*(((t>>3)*4 + (c>>5))*32 + (t&7)*4 + ((c>>3)&3)) + 2*(c&7)
 *   K,  8-bit (2048 B):  16*(((t>>3)*2 + (c>>6))*32 + (t&7)*4 + ((c>>4)&3)) + (c&15)
 *   K,  8-bit, 32-channel scale groups (2048 B; every tensor-core k-step inside one group):
 *                        16*(((t>>3)*2 + (c>>6))*32 + (t&7)*4 + ((c>>3)&3))
 *                        + 4*(2*((c>>5)&1) + ((c>>2)&1)) + (c&3)
 *   V, 16-bit (4096 B):  16*(32*(c>>4) + 4*(c&7) + ((t&7)>>1)) + 4*(2*(t>>3) + ((c>>3)&1)) + 2*(t&1)
 *   V,  8-bit (2048 B):  16*(32*(c>>5) + 4*(c&7) + ((t&7)>>1)) + 8*((c>>4)&1)
 *                        + 2*(2*(t>>3) + ((c>>3)&1)) + (t&1)
 *   witness (512 B, fp16 bits):  16*(4*(t&7) + (b>>2)) + 8*(t>>3) + 2*(b&3)
 *   scale   (32 B,  fp16 bits):  2*(2*(t&7) + (t>>3))
 *   scale, 32-channel groups (128 B, fp16 bits; group g = channels 32g..32g+31):
 *                        16*(t&7) + 4*g + 2*(t>>3)
 *   value witness (64 B, fp16 bits):  8*(t&7) + 4*k + 2*(t>>3), k = 0: rho^v_t =
 *                        ||v_hat_t - v_t||, k = 1: ||v_t|| (both rounded up; [W] Sec. 3,
 *                        the output bound ||y - y_hat|| <= 2 TV max_t ||v_t|| + sum_t p~_t rho^v_t)
 *   key outliers (fp16 bits, column col in 0..2m-1; column 2i holds channel pairs[i],
 *                 column 2i+1 channel pairs[i] + 64; unused columns 0):
 *       m <= 4 (256 B):  8*(4*(t&7) + (col>>1)) + 4*(t>>3) + 2*(col&1)
 *       m <= 8 (512 B):  16*(4*(t&7) + ((col&7)>>1)) + 8*(col>>3) + 4*(t>>3) + 2*(col&1)
 *     ([W] Sec. 6.2.5 fixed-channel outlier bypass: a fixed set of m RoPE pairs per
 *     (layer, kv head) is stored in fp16 (round to nearest even) and left out of the
 *     INT8 amax; the INT8 code of a bypassed channel is 0).  Head-major like the scales.
 * INT8 codes (both INT8 formats) are stored offset binary: the byte is code + 128
 * (code 0 is 0x80), so that the decode turns a byte into an fp16 operand with one
 * byte permute.
 * Band b holds the RoPE frequency pairs 4b..4b+3 of the half-split pairing
 * (pair j = channels j and j+64), i.e. channels 4b..4b+3 and 64+4b..64+4b+3
 * ([W] Sec. 4.1, eq. (2)).
 */
typedef struct kvq_cache {
  int32_t k_fmt;          /* kvq_fmt of the key plane                                  */
  int32_t v_fmt;          /* kvq_fmt of the value plane                                */
  int32_t num_kv_heads;   /* kv heads per layer                                        */
  int32_t num_pages;      /* pages in every plane                                      */
  int32_t layer;          /* layer index: a word of the dither counter                 */
  int32_t reserved;       /* must be 0                                                 */
  uint64_t dither_seed;   /* Philox key of the INT8 dither stream                      */
  void* k_data;           /* K tiles                                                   */
  void* v_data;           /* V tiles                                                   */
  uint16_t* k_scale;      /* K scale tiles (fp16 bits); non-NULL iff the K format has a scale */
  uint16_t* v_scale;      /* V scale tiles (fp16 bits); non-NULL iff the V format has a scale */
  uint16_t* witness;      /* witness tiles (fp16 bits); required by kvq_append, and by
                             kvq_decode_attn when the meter is on                      */
  uint16_t* v_witness;    /* value witness tiles (fp16 bits) or NULL; written by kvq_append
                             when non-NULL, required by kvq_decode_attn with KVQ_TIER_V */
  const int32_t* outlier_pairs; /* [num_kv_heads][n_outlier_pairs] RoPE pair indices j in 0..63
                             (channels j and j+64) bypassed in fp16, device memory; NULL iff
                             n_outlier_pairs == 0.  INT8-dithered keys only. */
  int32_t n_outlier_pairs;  /* m in 0..8 (0: no bypass); pairs of one head are distinct   */
  int32_t reserved2;        /* must be 0                                                 */
  uint16_t* k_outlier;      /* key outlier tiles (fp16 bits); non-NULL iff m > 0         */
} kvq_cache;

/* Meter configuration ([W] Sec. 4.2 request-level budget, Sec. 4.3 saturation). */
typedef struct kvq_meter_params {
  uint32_t tiers;     /* bit 0: Tier A witness bound; bit 1: Tier B dither certificate (INT8 keys only, either scale layout);
                         bit 2: value side of the output-error bound; bit 3: alternative bound shapes
                         (two-sided, det-tanh); bits 2 and 3 require Tier A                          */
  int32_t n_layers;   /* L in delta_loc = delta_req / (L * H * T)                                      */
  int32_t n_q_heads;  /* H (query heads)                                                               */
  int32_t n_steps;    /* T (decode steps the request budget covers; 256 in [W])                         */
  double delta_req;   /* request-level failure budget of Tier B                                        */
  float tau;          /* gate threshold for the coverage counts of kvq_meter                           */
  int32_t reserved;   /* must be 0                                                                     */
} kvq_meter_params;

#define KVQ_TIER_A 1u
#define KVQ_TIER_B 2u
#define KVQ_TIER_V 4u
#define KVQ_TIER_S 8u

/* Floats per (sequence, query head) cell of meter_state. */
#define KVQ_METER_STATE_FLOATS 8

/* Bytes of one tile of a plane: plane 0 = K, 1 = V, 2 = K scale, 3 = V scale, 4 = witness,
   5 = value witness, 6 = key outliers with m <= 4 pairs, 7 = key outliers with m <= 8 pairs.
   Returns 0 for a plane the format does not store. */
size_t kvq_tile_bytes(int32_t fmt, int32_t plane);

/* sizeof of the ABI structs as this library was compiled: which 0 = kvq_cache,
   1 = kvq_meter_params (0 for other values); lets bindings check their layouts. */
size_t kvq_sizeof(int32_t which);

/*
 * kvq_append -- quantize-on-append ([W] Sec. 4.2 "Subtractive dither",
 * Sec. 6.2.1 and 6.2.3; [C] "One kernel spans cartridge and live KV" for the
 * K16/V8 layout).
 *
 * k_dev, v_dev: [num_tokens][num_kv_heads][128] post-RoPE keys and values,
 *   element type in_dtype (KVQ_DTYPE_F32 or KVQ_DTYPE_BF16).
 * slot_mapping_dev: [num_tokens] int32 physical slot (page * 16 + offset) of
 *   each token; a negative slot skips the token.
 * For each (token, kv head) the kernel writes the K and V codes, the fp16
 * scales of scaled formats, and the 16 fp16 witness values: the band norms of
 * the key residual k_hat - k, rounded up ([W] Sec. 4.1, eq. (2)).  Scales:
 *   E4M3_SCALED: s = fp16_rn(fp32(amax / 448)),  code = e4m3_rn_satfinite(fp32(x / s))
 *   INT8_DITHER: s = fp16_rn(fp32(amax / 126.5)), code = clamp(rint(fp32(fp32(x / s) + xi)), -127, 127)
 *   INT8_DITHER_G32: the same per group of 32 channels (amax and s of channels 32g..32g+31; [W] Sec. 6.2.3)
 * (amax = 0 stores scale 0 and zero codes).  A cache whose keys are INT8_DITHER_G32 must have
 * INT8_DITHER_G32 values and vice versa, and has no outlier bypass (else KVQ_ERR_UNSUPPORTED_LAYOUT).  The dither xi comes from
 * Philox4x32-10 with key (seed low 32 bits, seed high 32 bits), counter
 * (slot, layer, kv_head, c >> 4), output word w = (c >> 2) & 3; the 8-bit
 * field f of channel c is byte (c & 3) of w (bits 8 (c & 3) .. 8 (c & 3) + 7),
 * and xi = f * 2^-8 - 1/2: a 256-point grid of [-1/2, 1/2) whose values
 * are exact in fp16, so the decode's fp16 operands carry exactly the xi used
 * here.  The K and V planes of a token share it ([W] Sec. 6.2.1, 6.2.3).
 * Device errors: KVQ_ERR_DEVICE_BOUNDS (slot beyond the cache; the token is
 * skipped), KVQ_ERR_NONFINITE_INPUT (non-finite input or fp16 scale overflow;
 * the token is written), KVQ_ERR_RANGE (a value scale above
 * KVQ_MAX_VALUE_SCALE; the token is written but decode would lose it).
 */
kvq_status kvq_append(const kvq_cache* cache, const void* k_dev, const void* v_dev, int32_t in_dtype,
                      const int32_t* slot_mapping_dev, int32_t num_tokens, int32_t* err_word_dev,
                      kvq_stream_t stream);

/*
 * kvq_append_rope -- kvq_append of keys that arrive pre-RoPE: the rotary position embedding is applied
 * on append ([W] Sec. 6.2.3 write path; [C] the cache keeps keys post-RoPE), and the rotated binary32
 * key is the exact key of the witness.
 * k_pre_dev: [num_tokens][num_kv_heads][128] pre-RoPE keys (in_dtype as for kvq_append).
 * positions_dev: [num_tokens] int32 absolute position of each token.
 * cos_sin_dev: [max_position][128] fp32, 16-byte aligned, caller-owned: at row p, cos(p theta_j) for
 *   j = 0..63, then sin(p theta_j), theta_j = theta^(-2j/128) (the model's cos/sin cache).
 * Half-split pairs (channel j with j + 64): x' = fl(fl(x c) - fl(y s)), y' = fl(fl(y c) + fl(x s)) in
 * binary32, each product and sum rounded once (no fused multiply-add).
 * Device errors: those of kvq_append, and KVQ_ERR_DEVICE_BOUNDS for a position outside
 * [0, max_position) (the token is skipped).
 */
kvq_status kvq_append_rope(const kvq_cache* cache, const void* k_pre_dev, const void* v_dev, int32_t in_dtype,
                           const int32_t* positions_dev, const float* cos_sin_dev, int32_t max_position,
                           const int32_t* slot_mapping_dev, int32_t num_tokens, int32_t* err_word_dev,
                           kvq_stream_t stream);

/* Workspace bytes kvq_decode_attn needs for (batch, num_kv_heads, num_q_heads) on the current device. */
size_t kvq_decode_workspace_size(int32_t batch, int32_t num_kv_heads, int32_t num_q_heads);

/*
 * kvq_decode_attn -- one decode step of one layer: split-KV paged GQA
 * attention over [shared prefix ++ live suffix] with one online-softmax state
 * per sequence and query head, the meter accumulated in the same pass, and a
 * log-sum-exp merge of the splits ([W] Sec. 6.2.2: the certificate, like the
 * output, is a p~-weighted average, so both merge under the same weights;
 * [C] "One kernel spans cartridge and live KV").
 *
 * cache: the layer's live paged cache.  prefix (nullable): a shared dense
 *   prefix of prefix_len tokens stored in pages 0, 1, ... of its own cache
 *   (same num_kv_heads); every sequence attends to it before its suffix.
 * q_dev: [batch][num_q_heads][128] post-RoPE queries (q_dtype F32 or BF16);
 *   query head h reads kv head h / (num_q_heads / num_kv_heads).
 * block_table_dev: [batch][max_pages_per_seq] int32 physical pages of each
 *   sequence's live suffix; seq_lens_dev: [batch] int32 live token counts.
 * sm_scale: softmax scale (1/sqrt(128) for standard attention).
 * meter (nullable => meter off): tiers to accumulate.  With the meter off the
 *   witness is not read and `out` is bit-identical to the meter-on output.
 * out_dev: [batch][num_q_heads][128] fp32 attention output sum_t p~_t v_hat_t.
 * meter_state_dev (nullable iff meter off): [batch][num_q_heads][8] fp32
 *   (KVQ_METER_STATE_FLOATS):
 *   [0] ln(A - 1) of Tier A, A = sum_t p~_t e^{c_t}, c_t = sm_scale *
 *       sum_b ||q_b|| w_{t,b} ([W] Thm. 1, Thm. 2); -inf when A = 1;
 *   [1] ln(A_B - 1) of Tier B, u_t = sm_scale s_t (||q|| sqrt(2 ln(2S/delta_loc)/12)
 *       + ||q||_1 2^-9) ([W] Sec. 4.2; the second term bounds the mean of the dithered
 *       rounding error on the 256-point dither grid); with 32-channel group scales
 *       u_t = sm_scale (kappa sqrt(sum_g ||q_g||^2 s_{g,t}^2) + 2^-9 sum_g ||q_g||_1 s_{g,t}),
 *       kappa = sqrt(2 ln(2S/delta_loc)/12); NaN when Tier B is off;
 *   [2] log-sum-exp of the compressed logits (natural log); [3] tokens attended S;
 *   [4] R = sum_t p~_t rho^v_t and [5] Vmax = max_t ||v_t|| from the value
 *       witness ([W] Sec. 3), NaN when KVQ_TIER_V is off (0 for an empty sequence);
 *   [6] max_t c_t and [7] 1 - A^- = sum_t p~_t (1 - e^{-c_t}) of Tier A's radii
 *       ([W] Sec. 4.3 Prop. 1 and the det-tanh shape), NaN when KVQ_TIER_S is off.
 * workspace_dev / ws_bytes: scratch of at least kvq_decode_workspace_size().
 * An empty sequence (no prefix, seq_len 0) yields out = 0 and ln(A-1) = -inf.
 * Returns KVQ_ERR_INVALID_ARG (nothing launched) when batch * num_kv_heads *
 * (prefix pages + max_pages_per_seq) exceeds 2^31 - 1: pages of the call are
 * indexed with 32-bit integers.
 */
kvq_status kvq_decode_attn(const kvq_cache* cache, const kvq_cache* prefix, int32_t prefix_len,
                           const void* q_dev, int32_t q_dtype, int32_t batch, int32_t num_q_heads,
                           const int32_t* block_table_dev, int32_t max_pages_per_seq,
                           const int32_t* seq_lens_dev, float sm_scale, const kvq_meter_params* meter,
                           float* out_dev, float* meter_state_dev, void* workspace_dev, size_t ws_bytes,
                           int32_t* err_word_dev, kvq_stream_t stream);

/*
 * kvq_decode_attn_append -- one decode step's append and attention in one
 * call: kvq_append of each sequence's newest token followed by
 * kvq_decode_attn.  The append runs as a small grid ahead of the decode; the
 * decode is launched as its programmatic dependent, runs alongside it, and
 * waits for it only before loading a page that holds a new token, so the
 * append costs no separate step on the GPU timeline ([W] Sec. 6.2.1: quantize
 * on write with the dither the read side regenerates).
 *
 * k_new_dev, v_new_dev: [batch][num_kv_heads][128] post-RoPE key and value of
 *   the newest token of each sequence, element type kv_dtype (KVQ_DTYPE_F32 or
 *   KVQ_DTYPE_BF16), 16-byte aligned.  The token is live position
 *   seq_lens[s] - 1 of sequence s; it is written at the slot the block table
 *   gives for that position (page block_table[s][(seq_lens[s] - 1) / 16],
 *   offset (seq_lens[s] - 1) % 16), exactly the bytes kvq_append would write
 *   for that slot, and is attended in the same call.  Sequences with
 *   seq_lens[s] == 0 append nothing.  The cache's witness plane is required.
 * Every other argument, output and error is that of kvq_decode_attn; input
 *   errors of the appended token are reported as kvq_append reports them
 *   (KVQ_ERR_NONFINITE_INPUT, KVQ_ERR_RANGE).
 */
kvq_status kvq_decode_attn_append(const kvq_cache* cache, const void* k_new_dev, const void* v_new_dev,
                                  int32_t kv_dtype, const kvq_cache* prefix, int32_t prefix_len,
                                  const void* q_dev, int32_t q_dtype, int32_t batch, int32_t num_q_heads,
                                  const int32_t* block_table_dev, int32_t max_pages_per_seq,
                                  const int32_t* seq_lens_dev, float sm_scale, const kvq_meter_params* meter,
                                  float* out_dev, float* meter_state_dev, void* workspace_dev, size_t ws_bytes,
                                  int32_t* err_word_dev, kvq_stream_t stream);

/* Optional outputs of kvq_decode_attn_ex. */
typedef struct kvq_decode_extras {
  float* page_log_contrib;  /* [batch][num_q_heads][contrib_stride] or NULL: per page of a sequence's
                               page list (the prefix pages, then the live pages) the natural log of
                               sum_{t in page} e^{x_t} (e^{c_t} - 1), x_t the compressed logit, c_t the
                               Tier A radius (-inf where every c_t is 0); exp(value - lse) is the page's
                               contribution to A - 1 ([W] Sec. 6.3.5: A decomposes over blocks and paging
                               in a block's exact values removes its contribution).  Requires the meter. */
  int32_t contrib_stride;   /* >= ceil(prefix_len / 16) + max_pages_per_seq                            */
  int32_t reserved;         /* must be 0                                                               */
} kvq_decode_extras;

/*
 * kvq_decode_attn_ex -- kvq_decode_attn_append with the newest tokens optional (k_new_dev and
 * v_new_dev both NULL: no append) and the optional outputs of `extras` (nullable).  Everything
 * else is that of kvq_decode_attn_append / kvq_decode_attn.
 */
kvq_status kvq_decode_attn_ex(const kvq_cache* cache, const void* k_new_dev, const void* v_new_dev, int32_t kv_dtype,
                              const kvq_cache* prefix, int32_t prefix_len, const void* q_dev, int32_t q_dtype,
                              int32_t batch, int32_t num_q_heads, const int32_t* block_table_dev,
                              int32_t max_pages_per_seq, const int32_t* seq_lens_dev, float sm_scale,
                              const kvq_meter_params* meter, const kvq_decode_extras* extras, float* out_dev,
                              float* meter_state_dev, void* workspace_dev, size_t ws_bytes, int32_t* err_word_dev,
                              kvq_stream_t stream);

/*
 * kvq_gate -- greedy block page-in plan from the page contributions ([W] Sec. 6.3.5, Sec. 6.1 "Gate"):
 * per (sequence, query head), the shortest list of pages, taken in decreasing order of contribution
 * (ties to the lower page index), whose removal brings A - 1 (the state's ln(A - 1)) down to
 * sqrt(1 + 2 tau) - 1, i.e. the meter 1/2 (A^2 - 1) to at most tau (the compressed distribution held
 * fixed, as on the page).
 * page_log_contrib_dev / contrib_stride: as written by kvq_decode_attn_ex; meter_state_dev:
 *   [batch][num_q_heads][8] of the same call; seq_lens_dev, prefix_len: that call's.  A sequence
 *   has ceil(prefix_len / 16) + ceil(seq_len / 16) pages; at most 16384.
 * n_page_in_dev: [batch][num_q_heads] int32, the list's length (0 when the meter is already <= tau).
 * page_list_dev (nullable): [batch][num_q_heads][max_list] int32, the first min(n, max_list) pages of
 *   the list in order, -1 after them.
 * A NaN contribution (non-finite inputs, which the decode reports in its error word) counts as none;
 * a cell whose ln(A - 1) is NaN gets the empty plan.
 */
kvq_status kvq_gate(const float* page_log_contrib_dev, int32_t contrib_stride, const float* meter_state_dev,
                    int32_t batch, int32_t num_q_heads, const int32_t* seq_lens_dev, int32_t prefix_len, float tau,
                    int32_t* n_page_in_dev, int32_t* page_list_dev, int32_t max_list, kvq_stream_t stream);

/*
 * kvq_zero_witness -- after a repair (the pages' exact values written back into the cache), zero
 * the witness (and the value witness, if the cache has one) of the repaired slots, so the meter
 * stops charging them ([W] Sec. 6.1: "write back, zero the witness").
 * slots_dev: [n] int32 physical slots; negative slots are skipped; a slot past the cache is reported
 * as KVQ_ERR_DEVICE_BOUNDS through err_word_dev (nullable).
 */
kvq_status kvq_zero_witness(const kvq_cache* cache, const int32_t* slots_dev, int32_t n, int32_t* err_word_dev,
                            kvq_stream_t stream);

/*
 * kvq_decode_attn_noalloc -- kvq_decode_attn without a caller-provided
 * workspace.  No counterpart on the source pages: it exists for callers that
 * cannot allocate device memory for scratch -- a plugin or embedding host
 * that owns every device allocation and passes the library only its inputs
 * and outputs, or a serving loop whose memory is planned up front and that
 * must not allocate on the request path.
 *
 * Arguments, outputs and device errors are those of kvq_decode_attn.  The
 * scratch is a file-scope device array of KVQ_STATIC_WORKSPACE_BYTES (16 MiB)
 * inside the library, which every GPU that loads the library holds until the
 * process exits.  The first call on a device looks up that array's device
 * address (with that device current); with lazy module loading that lookup may
 * also be when the driver loads the library's device code and reserves the
 * array, so on a device without 16 MiB free that first call can return
 * KVQ_ERR_CUDA.  Make the first call on each device at start-up, before any
 * stream capture.  The address is kept for the life of the process: a device
 * reset (cudaDeviceReset) invalidates it, and the library does not support
 * this entry point after one.  Calls whose workspace need
 * (kvq_decode_workspace_size) exceeds KVQ_STATIC_WORKSPACE_BYTES return
 * KVQ_ERR_WORKSPACE_TOO_SMALL without enqueuing work.  The call itself
 * allocates nothing (no cudaMalloc / cudaFree, no allocating library call).
 * All calls share the one array and it keeps the last call's contents; the
 * decode writes every scratch value before reading it, so nothing needs
 * clearing between calls.  Calls that overlap on the GPU (different streams,
 * or different host threads) race on the array: serialise them.
 */
#define KVQ_STATIC_WORKSPACE_BYTES (16u << 20)
kvq_status kvq_decode_attn_noalloc(const kvq_cache* cache, const kvq_cache* prefix, int32_t prefix_len,
                                   const void* q_dev, int32_t q_dtype, int32_t batch, int32_t num_q_heads,
                                   const int32_t* block_table_dev, int32_t max_pages_per_seq,
                                   const int32_t* seq_lens_dev, float sm_scale, const kvq_meter_params* meter,
                                   float* out_dev, float* meter_state_dev, int32_t* err_word_dev,
                                   kvq_stream_t stream);

/*
 * kvq_meter -- meter finalisation and telemetry on the device ([W] Sec. 4.3;
 * Sec. 6.2.4 "Certificate telemetry in production": aggregate on the GPU,
 * count non-finite values separately).
 *
 * meter_state_dev: [n_layers][batch][num_q_heads][8] as written by kvq_decode_attn.
 * meter_a_dev:  [n_layers][batch][num_q_heads] min(1, 1/2 (A^2 - 1)) of Tier A.
 * raw_a_dev:    same shape, the raw log score ln(1/2 (A^2 - 1)) (finite for finite inputs).
 * cert_b_dev (nullable): same shape, min(1, 1/2 (A_B^2 - 1)).
 * out_bound_dev (nullable): same shape, the output-error bound 2 meter_a Vmax + R
 *   of ||y - y_hat|| ([W] Sec. 3 with Tier A's meter for TV); NaN where the state
 *   has no value side.
 * two_sided_dev (nullable): same shape, min(meter_a, 1/2 (A/A^- - A^-/A)) ([W] Sec. 4.3
 *   Prop. 1: neither form dominates, so the minimum); NaN without KVQ_TIER_S.
 * tanh_dev (nullable): same shape, tanh(max_t c_t) (TV <= tanh(max |eps|)); NaN without KVQ_TIER_S.
 * counts_dev:   int32[4]: cells with meter_a < tau, cells with cert_b < tau,
 *               non-finite cells, total cells (zeroed and filled by the call).
 * ranking_dev (nullable): [batch][n_layers * num_q_heads] int32 flat cell
 *   indices (layer * num_q_heads + head) of each request, highest raw score
 *   first, ties to the lower index (requires n_layers * num_q_heads <= 8192).
 */
kvq_status kvq_meter(const float* meter_state_dev, int32_t n_layers, int32_t batch, int32_t num_q_heads,
                     const kvq_meter_params* meter, float* meter_a_dev, float* raw_a_dev, float* cert_b_dev,
                     float* out_bound_dev, float* two_sided_dev, float* tanh_dev, int32_t* counts_dev,
                     int32_t* ranking_dev, kvq_stream_t stream);

/* Test hook: the dither xi of (seed, layer, kv_head, slots[i], channel c) into xi_dev[i * 128 + c]. */
kvq_status kvq_debug_dither(uint64_t seed, int32_t layer, int32_t kv_head, const int32_t* slots_dev, int32_t n,
                            float* xi_dev, kvq_stream_t stream);

/* Test hook: the device conversions kvq_append uses, applied to n fp32 values.
   kind 0: bf16 RNE (uint16 out); 1: e4m3 RNE satfinite (uint8 out); 2: fp16 RNE
   (uint16 out); 3: fp16 round-up (uint16 out). */
kvq_status kvq_debug_encode(int32_t kind, const float* x_dev, int64_t n, void* out_dev, kvq_stream_t stream);

/* Test hook: one warp runs the decode kernel's bounded wait (at most limit_ns <= 2 s of wall clock)
   on an mbarrier that nothing completes, then writes KVQ_ERR_TIMEOUT to err_word_dev; the context
   stays usable.  Exercises the failure path without faulting or hanging the GPU. */
kvq_status kvq_debug_wait_timeout(uint64_t limit_ns, int32_t* err_word_dev, kvq_stream_t stream);

/* Measurement hook: while set (both non-NULL, cudaEvent_t handles), every decode call made from
   this host thread records start_event immediately before the decode kernel's launch and
   stop_event immediately after it, on the call's stream, so the kernel's own duration can be timed
   apart from the append and merge launches around it (a fused call then launches the decode after
   its append instead of overlapping them).  NULL, NULL clears it. */
kvq_status kvq_debug_time_decode(void* start_event, void* stop_event);

/* Human-readable name of a status code (static storage). */
const char* kvq_status_string(int32_t status);

/* KVQ_VERSION of the loaded library. */
int32_t kvq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H_ */
