/*
 * qwen35_decode.h — C ABI of the GB300 (sm_103a) single-token decode library for
 * Qwen3.5 decoder layers: the gated full-attention layer and the Gated DeltaNet
 * (linear-attention) layer.
 *
 * The calls follow the problem statement of the pages "full_attention.rs"
 * (forward_full_attention: config, layer weights, scratch, KV cache, x_in,
 * cache_pos, seq_len_attn, stream) and "linear_attention.rs"
 * (forward_linear_attention: config, layer weights, persistent conv/SSM state,
 * scratch, x_in, stream), with the structs of "mod.rs".
 *
 * Conventions for every call:
 *  - All tensor pointers are DEVICE pointers unless a comment says otherwise, and
 *    must be 16-byte aligned. bf16 values travel as uint16_t bit patterns.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream). Calls only enqueue
 *    work: they never synchronise, except qwen35_read_device_status.
 *  - The caller owns and allocates everything (weights, caches, states, scratch);
 *    the library allocates nothing on the forward path and keeps no pointer after
 *    a call returns (a captured graph keeps them: see qwen35_graph_create).
 *  - Return value: QWEN35_OK or an error code. Argument errors are reported
 *    before anything is enqueued. Errors of asynchronous device work surface at the
 *    caller's next synchronisation (CUDA error) or in the device status word.
 *  - Device status word: the first 4 bytes of every scratch buffer hold an int32
 *    status that kernels set (never clear) when a bounded wait gives up
 *    (QWEN35_ERR_DEVICE_TIMEOUT) or a device-resident position is out of range
 *    (QWEN35_ERR_DEVICE_RANGE; that kernel then skips its work). The caller zeroes
 *    it when the scratch is created (qwen35_scratch_init) and may read it with
 *    qwen35_read_device_status.
 */
#ifndef QWEN35_DECODE_H
#define QWEN35_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define QWEN35_API __attribute__((visibility("default")))
#else
#define QWEN35_API
#endif

typedef uint16_t qwen35_bf16;

enum qwen35_status {
    QWEN35_OK = 0,
    QWEN35_ERR_INVALID_ARGUMENT = 1, /* null/misaligned pointer, bad dims, scratch too small */
    QWEN35_ERR_OUT_OF_RANGE = 2,     /* cache_pos >= capacity, seq_len_attn not in [1, cache_pos+1] */
    QWEN35_ERR_UNSUPPORTED = 3,      /* dims beyond the compiled kernels' limits */
    QWEN35_ERR_CUDA = 4,             /* a CUDA runtime call or launch failed */
    QWEN35_ERR_DEVICE_TIMEOUT = 5,   /* device status only: a bounded wait gave up */
    QWEN35_ERR_DEVICE_RANGE = 6      /* device status only: device position out of range */
};

enum qwen35_layer_kind {
    QWEN35_LAYER_FULL_ATTENTION = 0,
    QWEN35_LAYER_LINEAR_ATTENTION = 1
};

/* Dimensions of a checkpoint: the Qwen35ForwardConfig struct of "mod.rs" (its 4B
 * preset is qwen3_5_4b_mlx_int8). vocab is carried but unused (no embedding or
 * lm_head here). group_size must be 64. */
typedef struct qwen35_config {
    uint32_t hidden, intermediate, num_layers, vocab, group_size;
    float rms_eps;
    uint32_t num_heads, num_kv_heads, head_dim;
    float rope_theta;
    uint32_t rotary_dim;
    uint32_t num_k_heads_lin, num_v_heads_lin, k_head_dim_lin, v_head_dim_lin;
    uint32_t conv_kernel_size;
} qwen35_config;

/* An int8 group-64 affine matrix W [n][k] (the QuantWeights type the pages use;
 * its format is not printed there, this is the MLX-8bit layout):
 *   codes  uint8 [n][k] row-major;
 *   scales bf16  [n][gstride], biases bf16 [n][gstride], gstride = round_up(k/64, 8)
 *   (the padding keeps every row 16-byte aligned; padded entries are never read);
 *   W[r][c] = scales[r][c/64] * codes[r][c] + biases[r][c/64].
 * k must be a multiple of 64 and at most 12288. Borrowed, never written. */
typedef struct qwen35_qweight {
    const uint8_t* codes;
    const qwen35_bf16* scales;
    const qwen35_bf16* biases;
    uint32_t n, k;
} qwen35_qweight;

/* Full-attention layer weights (FullAttentionLayer, "mod.rs"). Norm vectors are
 * bf16: input_ln/post_ln [hidden], q_norm/k_norm [head_dim]. q_proj is
 * [2*num_heads*head_dim][hidden] with each head's rows ordered [Q_h | gate_h];
 * k_proj, v_proj [num_kv_heads*head_dim][hidden]; o_proj [hidden][num_heads*head_dim];
 * gate_proj, up_proj [intermediate][hidden]; down_proj [hidden][intermediate]. */
typedef struct qwen35_fa_layer {
    const qwen35_bf16 *input_ln, *q_norm, *k_norm, *post_ln;
    qwen35_qweight q_proj, k_proj, v_proj, o_proj, gate_proj, up_proj, down_proj;
} qwen35_fa_layer;

/* Linear-attention layer weights (LinearAttentionLayer, "mod.rs"): a_log fp32
 * [Hv]; dt_bias bf16 [Hv]; conv1d_weight bf16 [C][conv_kernel_size] with
 * C = 2*Hk*Dk + Hv*Dv; norm_weight bf16 [Dv]; in_proj_a/b [Hv][hidden];
 * in_proj_qkv [C][hidden] with channels ordered [Q | K | V]; in_proj_z
 * [Hv*Dv][hidden]; out_proj [hidden][Hv*Dv]; MLP as in the full-attention layer. */
typedef struct qwen35_gdn_layer {
    const qwen35_bf16* input_ln;
    const float* a_log;
    const qwen35_bf16 *dt_bias, *conv1d_weight;
    qwen35_qweight in_proj_a, in_proj_b, in_proj_qkv, in_proj_z;
    const qwen35_bf16* norm_weight;
    qwen35_qweight out_proj;
    const qwen35_bf16* post_ln;
    qwen35_qweight gate_proj, up_proj, down_proj;
} qwen35_gdn_layer;

/* KV cache of one full-attention layer and one sequence (LayerKvCache, "mod.rs"),
 * in one of two formats (MetalKvDtype there):
 *  - QWEN35_KV_BF16 (0): k and v are bf16 [capacity][num_kv_heads][head_dim];
 *    k_scales, v_scales unused (may be NULL).
 *  - QWEN35_KV_TURBO8 (1): the Turbo8 format, in the WHT-rotated basis (the
 *    forward rotates k and v before the append, q before attention and the output
 *    back after it): k and v are FP8 E4M3 codes, uint8 [capacity][num_kv_heads]
 *    [head_dim]; k_scales and v_scales are bf16 [capacity][sstride], one scale per
 *    16 consecutive elements of a token's row (element j of kv-head g uses scale
 *    g * head_dim / 16 + j / 16), sstride = round_up(num_kv_heads * head_dim / 16, 8)
 *    (the pages keep the scales unpadded; the padding keeps every token's row of
 *    scales 16-byte aligned for the bulk copies). 1.125 bytes per element.
 * A forward writes exactly row cache_pos of each array and reads rows
 * [0, seq_len_attn). All pointers 16-byte aligned.
 *
 * Paged (optional; the production decode path the module page names, whose format
 * the pages do not print): with block_table non-NULL, k and v are pools of blocks
 * of block_tokens token rows, bf16 [num_blocks][block_tokens][num_kv_heads]
 * [head_dim], and logical token t lives in row t % block_tokens of pool block
 * block_table[t / block_tokens] (int32, in [0, num_blocks); the caller keeps it
 * valid for every block a forward touches: [0, seq_len_attn) and cache_pos).
 * capacity counts logical tokens and is a multiple of block_tokens; block_tokens
 * is a power of two, at least 8. bf16 only. A batch of caches shares one pool:
 * sequence b's table is block_table + b * (capacity / block_tokens). With
 * block_table NULL (block_tokens ignored) the rows are contiguous as above. */
enum qwen35_kv_dtype {
    QWEN35_KV_BF16 = 0,
    QWEN35_KV_TURBO8 = 1
};
typedef struct qwen35_kv_cache {
    void* k;
    void* v;
    uint32_t capacity;
    uint32_t dtype;
    qwen35_bf16* k_scales;
    qwen35_bf16* v_scales;
    const int32_t* block_table;
    uint32_t block_tokens;
    uint32_t reserved;
} qwen35_kv_cache;

/* Persistent state of one linear-attention layer (LinearAttentionState,
 * "mod.rs"): conv_state fp32 [C][conv_kernel_size] (newest input in the last
 * slot); gdn_state fp32, the per-head Dk x Dv matrices S_h stored in column
 * blocks of 32: [Hv][Dv/32][Dk][32], S_h[k][v] at
 * ((h * (Dv/32) + v/32) * Dk + k) * 32 + v % 32 (each block is the contiguous
 * working set of one CTA). Caller-allocated and zeroed before the first token;
 * updated in place by every forward. */
typedef struct qwen35_gdn_state {
    float* conv_state;
    float* gdn_state;
} qwen35_gdn_state;

/* One layer of a decode stack: kind selects fa+kv or gdn+state. */
typedef struct qwen35_layer {
    int32_t kind;
    const qwen35_fa_layer* fa;
    const qwen35_kv_cache* kv;
    const qwen35_gdn_layer* gdn;
    const qwen35_gdn_state* state;
} qwen35_layer;

/* Once per process and device, before any forward: queries the device and sets
 * kernel attributes (the counterpart of Qwen35Kernels::resolve in "mod.rs",
 * which looks every kernel up once at startup). Returns QWEN35_ERR_CUDA without a
 * usable sm_103 device. */
QWEN35_API int qwen35_init(void);

/* Static description of a status code (never NULL). */
QWEN35_API const char* qwen35_status_string(int status);

/* Bytes of scratch a forward of `layer_kind` needs (the FullAttentionScratch /
 * LinearAttentionScratch buffers of "mod.rs", plus the device status word and the
 * split-KV attention partials). qwen35_stack_scratch_bytes covers every layer of a
 * stack. 0 for an invalid config. */
QWEN35_API size_t qwen35_scratch_bytes(const qwen35_config* cfg, int layer_kind);
QWEN35_API size_t qwen35_stack_scratch_bytes(const qwen35_config* cfg);

/* Zero the device status word and the internal counters of a scratch buffer
 * (enqueued on `stream`). Call once after allocating scratch. */
QWEN35_API int qwen35_scratch_init(void* scratch, size_t scratch_bytes, void* stream);

/* Synchronise `stream`, then copy the device status word of `scratch` into
 * *host_status (host pointer). */
QWEN35_API int qwen35_read_device_status(const void* scratch, int32_t* host_status, void* stream);

/* Single-token full-attention decoder forward ("full_attention.rs",
 * forward_full_attention): input RMSNorm, q_proj with its [Q_h | gate_h] split,
 * k/v projections, per-head q/k RMSNorm, RoPE on the first rotary_dim dims at
 * position cache_pos, KV append at row cache_pos, GQA attention over tokens
 * [0, seq_len_attn), sigmoid(gate) gating, o_proj, residual + post RMSNorm, and the
 * SiLU-gated MLP with its residual. x_in, x_out: bf16 [hidden]; x_out may equal
 * x_in (no other aliasing). Errors: INVALID_ARGUMENT, OUT_OF_RANGE
 * (cache_pos >= kv->capacity, seq_len_attn == 0 or > cache_pos + 1), UNSUPPORTED
 * (head_dim not 64/128/256, rotary_dim odd or > head_dim, num_kv_heads > 8), CUDA. */
QWEN35_API int qwen35_forward_full_attention(const qwen35_config* cfg, const qwen35_fa_layer* layer,
                                  void* scratch, size_t scratch_bytes,
                                  const qwen35_kv_cache* kv,
                                  const qwen35_bf16* x_in, qwen35_bf16* x_out,
                                  uint32_t cache_pos, uint32_t seq_len_attn, void* stream);

/* The same forward with the position in device memory, for graph capture:
 * cache_pos = *d_cache_pos, seq_len_attn = cache_pos + 1, read by the kernels when
 * they run. The split-KV work partition is sized for max_seq_len tokens at
 * enqueue time. A device position outside [0, min(capacity, max_seq_len)) sets
 * QWEN35_ERR_DEVICE_RANGE in the status word and the layer's attention is skipped. */
QWEN35_API int qwen35_forward_full_attention_dpos(const qwen35_config* cfg, const qwen35_fa_layer* layer,
                                       void* scratch, size_t scratch_bytes,
                                       const qwen35_kv_cache* kv,
                                       const qwen35_bf16* x_in, qwen35_bf16* x_out,
                                       const int32_t* d_cache_pos, uint32_t max_seq_len,
                                       void* stream);

/* Single-token Gated DeltaNet decoder forward ("linear_attention.rs",
 * forward_linear_attention): input RMSNorm, in_proj_a/b/qkv/z, causal conv1d
 * update + SiLU with per-head L2 norm on the Q/K channels, gate =
 * exp(softplus(dt + dt_bias) * -exp(A_log)), beta = sigmoid(b), the gated
 * delta-rule state update and readout scaled by 1/sqrt(k_head_dim_lin), the
 * per-head RMSNorm gated by silu(z), out_proj, residual + post RMSNorm and the MLP.
 * The page copies x_final into a separate x_buf; here the last kernel writes x_out
 * directly, and x_out may equal x_in. Errors: INVALID_ARGUMENT, UNSUPPORTED
 * (k/v head dims not 32/64/128, num_v_heads_lin % num_k_heads_lin != 0), CUDA. */
QWEN35_API int qwen35_forward_linear_attention(const qwen35_config* cfg, const qwen35_gdn_layer* layer,
                                    void* scratch, size_t scratch_bytes,
                                    const qwen35_gdn_state* state,
                                    const qwen35_bf16* x_in, qwen35_bf16* x_out, void* stream);

/* The linear-attention forward above for callers that cannot allocate device
 * memory: a plug-in that lives inside a host framework which owns every device
 * allocation, a process whose memory budget is fixed once at start-up, or a
 * latency-critical path where cudaMalloc's device-wide synchronisation is not
 * acceptable. No counterpart on the pages (their forwards take caller-owned
 * scratch); it exists for those callers only.
 * Instead of caller scratch it uses one static device array of 256 KiB inside
 * the library (QWEN35_STATIC_SCRATCH_BYTES), which every GPU that loads the
 * library keeps until the process exits. Configs whose linear-attention scratch
 * (qwen35_scratch_bytes) exceeds it are rejected with QWEN35_ERR_UNSUPPORTED.
 * The first call on a device looks the array's device address up (once per
 * device, with that device current); make that first call before any stream
 * capture. Every call shares the array and each accepted call clears its status
 * word first, so calls whose work overlaps on the GPU (other streams, other host
 * threads) race on it: serialise them. Every argument is checked before the
 * device is touched: a rejected call enqueues nothing and leaves the previous
 * call's status word as it was. Arguments and errors otherwise as
 * qwen35_forward_linear_attention. Allocates nothing (no cudaMalloc/cudaFree). */
#define QWEN35_STATIC_SCRATCH_BYTES (256u * 1024u)
QWEN35_API int qwen35_forward_linear_attention_static(const qwen35_config* cfg,
                                                      const qwen35_gdn_layer* layer,
                                                      const qwen35_gdn_state* state,
                                                      const qwen35_bf16* x_in, qwen35_bf16* x_out,
                                                      void* stream);
/* The device status word of that static array (as qwen35_read_device_status is
 * for caller scratch): synchronises `stream`, then copies the status the last
 * qwen35_forward_linear_attention_static call on the current device left (0 if
 * none ran) into *host_status (host pointer). Allocates nothing. */
QWEN35_API int qwen35_read_static_status(int32_t* host_status, void* stream);

/* One decode step of a layer stack: layer i's output is layer i+1's input (the
 * caller's layer loop, which the module page leaves to the caller). Full-attention
 * layers use the device position *d_cache_pos (as in the _dpos forward); after
 * the last layer the kernel advances *d_cache_pos by one, so the same enqueued
 * sequence (or a graph of it) decodes consecutive tokens. x_in [hidden] is read by
 * layer 0; x_out [hidden] receives every layer's output in turn (it may equal
 * x_in). Scratch: qwen35_stack_scratch_bytes. */
QWEN35_API int qwen35_decode_step(const qwen35_config* cfg, const qwen35_layer* layers, uint32_t num_layers,
                       void* scratch, size_t scratch_bytes,
                       const qwen35_bf16* x_in, qwen35_bf16* x_out,
                       int32_t* d_cache_pos, uint32_t max_seq_len, void* stream);

/* A CUDA graph of one qwen35_decode_step, captured on `stream` (which must not be
 * capturing already). The graph keeps every pointer given here: the buffers must
 * outlive it. Replaying it decodes one token and advances *d_cache_pos. */
typedef struct qwen35_graph qwen35_graph;
QWEN35_API int qwen35_graph_create(const qwen35_config* cfg, const qwen35_layer* layers, uint32_t num_layers,
                        void* scratch, size_t scratch_bytes,
                        const qwen35_bf16* x_in, qwen35_bf16* x_out,
                        int32_t* d_cache_pos, uint32_t max_seq_len, void* stream,
                        qwen35_graph** out_graph);
QWEN35_API int qwen35_graph_launch(qwen35_graph* graph, void* stream);
QWEN35_API int qwen35_graph_destroy(qwen35_graph* graph);

/* Several independent sequences decoded in one step (multi-sequence decode: each
 * sequence has its own position, KV caches and linear-attention states; the
 * weights are shared and streamed from HBM once per step, the batch's later
 * passes over a layer's weights being served from L2). Every phase of the
 * stack runs for the batch's sequences back to back, so the grid barriers are
 * shared by the batch.
 *  - batch: 1..8 sequences.
 *  - x_in, x_out: [batch][hidden]; d_cache_pos: [batch] int32 (each advanced by
 *    one after the last layer); max_seq_len bounds every sequence's position.
 *  - layers: as for qwen35_decode_step, with every cache holding the batch's
 *    sequences contiguously, sequence b at the given pointer plus b times one
 *    sequence's size: kv->k and kv->v [batch][capacity][Hkv][D] (capacity shared;
 *    a paged cache: one shared pool, tables [batch][capacity / block_tokens]);
 *    conv_state [batch][C][conv_kernel_size]; gdn_state [batch][Hv][Dv/32][Dk][32].
 *  - scratch: qwen35_stack_scratch_bytes_batched(cfg, batch).
 * Errors as qwen35_decode_step; batch outside 1..8 is INVALID_ARGUMENT. Sequence b
 * computes exactly what qwen35_decode_step computes for it alone. */
QWEN35_API size_t qwen35_stack_scratch_bytes_batched(const qwen35_config* cfg, uint32_t batch);
QWEN35_API int qwen35_decode_step_batched(const qwen35_config* cfg, const qwen35_layer* layers,
                       uint32_t num_layers, uint32_t batch, void* scratch, size_t scratch_bytes,
                       const qwen35_bf16* x_in, qwen35_bf16* x_out,
                       int32_t* d_cache_pos, uint32_t max_seq_len, void* stream);
/* One layer for a batch of independent sequences (the per-layer forwards above,
 * several sequences at once; the layer's weights are streamed once, the batch's
 * projections run on the tensor cores): sequence b computes exactly what the
 * single-sequence forward computes for it.
 *  - batch: 1..8; x_in, x_out [batch][hidden] (x_out may equal x_in);
 *  - full attention: kv->k, kv->v [batch][capacity][Hkv][D] (paged: one pool,
 *    tables [batch][capacity / block_tokens]); d_cache_pos [batch]
 *    int32 in device memory, sequence b appending at d_cache_pos[b] and attending
 *    over d_cache_pos[b] + 1 tokens (read when the kernel runs, not advanced); a
 *    position outside [0, min(capacity, max_seq_len)) sets QWEN35_ERR_DEVICE_RANGE
 *    in the status word and that sequence's attention is skipped;
 *  - linear attention: conv_state [batch][C][conv_kernel_size], gdn_state
 *    [batch][Hv][Dv/32][Dk][32];
 *  - scratch: qwen35_stack_scratch_bytes_batched(cfg, batch) suffices.
 * Errors as the single-sequence forwards; batch outside 1..8 is INVALID_ARGUMENT. */
QWEN35_API int qwen35_forward_full_attention_batched(const qwen35_config* cfg, const qwen35_fa_layer* layer,
                                                     uint32_t batch, void* scratch, size_t scratch_bytes,
                                                     const qwen35_kv_cache* kv, const qwen35_bf16* x_in,
                                                     qwen35_bf16* x_out, const int32_t* d_cache_pos,
                                                     uint32_t max_seq_len, void* stream);
QWEN35_API int qwen35_forward_linear_attention_batched(const qwen35_config* cfg, const qwen35_gdn_layer* layer,
                                                       uint32_t batch, void* scratch, size_t scratch_bytes,
                                                       const qwen35_gdn_state* state, const qwen35_bf16* x_in,
                                                       qwen35_bf16* x_out, void* stream);
/* A CUDA graph of one qwen35_decode_step_batched (as qwen35_graph_create). */
QWEN35_API int qwen35_graph_create_batched(const qwen35_config* cfg, const qwen35_layer* layers,
                        uint32_t num_layers, uint32_t batch, void* scratch, size_t scratch_bytes,
                        const qwen35_bf16* x_in, qwen35_bf16* x_out,
                        int32_t* d_cache_pos, uint32_t max_seq_len, void* stream,
                        qwen35_graph** out_graph);

/* Multi-token prefill: the n_tokens tokens of a prompt through a layer (or a
 * stack) in one call, the step before decode that the module page "Module
 * qwen3_5" leaves out of the single-token path (its non-goals: multi-token
 * prefill). Token t of the prompt sits at position cache_pos + t and computes
 * exactly what the single-token forward computes for it after tokens 0 .. t-1
 * (full attention: append at cache_pos + t, attention over cache_pos + t + 1
 * tokens; linear attention: the conv and delta-rule states advanced token by
 * token), so a prefill of n tokens equals n single-token calls in order, up to
 * the rounding below.
 *  - x_in, x_out: bf16 [n_tokens][hidden] (x_out may equal x_in); every token's
 *    output is written.
 *  - Projections run as tensor-core GEMMs over all tokens at once, each GEMM
 *    input a bf16 vector. The projections whose outputs are kept (k_proj and
 *    v_proj fill the KV cache; in_proj_qkv, in_proj_a, in_proj_b drive the conv
 *    and delta-rule states) multiply each dequantised weight w = scale * code +
 *    bias as the sum of two bf16 values (bf16(w) + bf16(w - bf16(w)): w to 2^-16
 *    relative), so the caches and states match the single-token path's; the
 *    others multiply bf16(w) (relative 2^-9 per weight). The inputs the
 *    single-token path keeps unrounded inside its fused kernels (SiLU(gate) * up
 *    before down_proj, SiLU(z) * y_norm before out_proj) are rounded to bf16
 *    here. Both stay far inside the layer tolerance.
 *  - KV cache: bf16 (contiguous or paged) or Turbo8 (rows rotated and quantised
 *    as the single-token forward does); logical rows [cache_pos, cache_pos +
 *    n_tokens) are written, rows [0, cache_pos) read (a paged cache's table must
 *    name every block of [0, cache_pos + n_tokens)); cache_pos + n_tokens >
 *    capacity is QWEN35_ERR_OUT_OF_RANGE.
 *  - Scratch: qwen35_prefill_scratch_bytes(cfg, max_tokens) for any n_tokens up to
 *    max_tokens (its first 4 bytes are the device status word, as for decode);
 *    at most 65536 tokens per call.
 *  - The stack form runs layer i on layer i-1's output, all at positions
 *    cache_pos .. cache_pos + n_tokens - 1 (nothing is advanced in device memory).
 * Errors: INVALID_ARGUMENT (null or misaligned pointer, n_tokens 0 or above 65536,
 * scratch too small, shape mismatch), OUT_OF_RANGE, UNSUPPORTED (as for the
 * single-token forwards, and for full attention num_heads / num_kv_heads other
 * than 1, 2, 4 or 8), CUDA. Every argument is checked before anything is enqueued;
 * calls only enqueue work on `stream`. */
QWEN35_API size_t qwen35_prefill_scratch_bytes(const qwen35_config* cfg, uint32_t max_tokens);
QWEN35_API int qwen35_prefill_full_attention(const qwen35_config* cfg, const qwen35_fa_layer* layer,
                                             void* scratch, size_t scratch_bytes, const qwen35_kv_cache* kv,
                                             const qwen35_bf16* x_in, qwen35_bf16* x_out, uint32_t cache_pos,
                                             uint32_t n_tokens, void* stream);
QWEN35_API int qwen35_prefill_linear_attention(const qwen35_config* cfg, const qwen35_gdn_layer* layer,
                                               void* scratch, size_t scratch_bytes, const qwen35_gdn_state* state,
                                               const qwen35_bf16* x_in, qwen35_bf16* x_out, uint32_t n_tokens,
                                               void* stream);
QWEN35_API int qwen35_prefill_step(const qwen35_config* cfg, const qwen35_layer* layers, uint32_t num_layers,
                                   void* scratch, size_t scratch_bytes, const qwen35_bf16* x_in,
                                   qwen35_bf16* x_out, uint32_t cache_pos, uint32_t n_tokens, void* stream);

/* The prefill's projection on its own: Y[t][r] = bf16(sum_c W[r][c] X[t][c]) for
 * t < n_tokens, r < w->n, with w = scales[r][c/64] * codes[r][c] + biases[r][c/64]
 * taken as W = bf16(w) + bf16(w - bf16(w)) (w to 2^-16 relative) when exact is
 * nonzero, else as W = bf16(w); fp32 accumulation on the tensor cores. X bf16
 * [n_tokens][k], Y bf16 [n_tokens][n], device pointers, 16-byte aligned; scratch:
 * at least 256 bytes (its status word); with QWEN35_PREFILL_GEMM_SPLIT_SCRATCH
 * bytes or more, a GEMM whose 128-row x 256-token tiles would leave SMs idle
 * splits K over more CTAs (fp32 partial sums in the scratch, added in a fixed
 * order). Errors: INVALID_ARGUMENT, CUDA. */
#define QWEN35_PREFILL_GEMM_SPLIT_SCRATCH (256u + 152u * 128u * 256u * 4u)
QWEN35_API int qwen35_prefill_gemm(const qwen35_qweight* w, const qwen35_bf16* X, qwen35_bf16* Y,
                                   uint32_t n_tokens, int exact, void* scratch, size_t scratch_bytes,
                                   void* stream);

/* The quantised GEMV on its own (QuantWeights::gemv): y[n] = bf16(W x), x bf16 [k]. */
QWEN35_API int qwen35_gemv(const qwen35_qweight* w, const qwen35_bf16* x, qwen35_bf16* y, void* scratch,
                size_t scratch_bytes, void* stream);

/* The model's output head after the last decoder layer, with greedy token choice.
 * The pages stop at the decoder layers and leave the final norm, the lm_head and
 * sampling to the caller (page "Module qwen3_5": non-goals); this entry is that
 * tail in the pages' conventions:
 *   x_norm = bf16(RMSNorm(x) * final_norm), eps = cfg->rms_eps (as every rms_norm);
 *   logits[v] = bf16(sum_k W[v][k] x_norm[k]) for v < lm_head->n (the vocabulary);
 *   *token = the index of the largest logit, the lowest index among equal ones
 *            (NaN logits are never chosen; -1 if every logit is NaN).
 * x, final_norm: bf16 [hidden]; lm_head: [vocab][hidden] in the QuantWeights format
 * of qwen35_qweight (k = hidden, a multiple of 64, at most 12288); logits: bf16
 * [vocab], written; token: one int32 in device memory, written. All device
 * pointers, caller-owned, 16-byte aligned (token 4-byte aligned); scratch: at least
 * 256 bytes (its status word and barrier counter). Runs the quantised GEMV with
 * the norm in its prologue, then a one-block argmax, on `stream`. Errors:
 * QWEN35_ERR_INVALID_ARGUMENT (null or misaligned pointer, shape mismatch),
 * QWEN35_ERR_UNSUPPORTED (hidden > 12288), QWEN35_ERR_CUDA (launch failure). */
QWEN35_API int qwen35_lm_head_greedy(const qwen35_config* cfg, const qwen35_bf16* final_norm,
                                     const qwen35_qweight* lm_head, const qwen35_bf16* x, qwen35_bf16* logits,
                                     int32_t* token, void* scratch, size_t scratch_bytes, void* stream);

/* Byte offset inside a layer's scratch of a named intermediate the last forward of
 * that kind left there, or (size_t)-1 for an unknown name: the counterpart of the
 * intra_dump hook of "linear_attention.rs" (named buffers readable after a stream
 * synchronise). For a stack (qwen35_decode_step) the offsets of
 * qwen35_debug_stack_scratch_offset apply instead; both hold the last layer of
 * that kind's values.
 * Results handed between the kernel's CTAs are 32-bit words, one per element, the
 * bf16 value in the HIGH 16 bits (the low 16 bits are internal):
 *   full attention:   q_full [2*H*D], k, v [Hkv*D], gated_attn [H*D], o, x_resid [hidden],
 *                     gate_act, up_act [intermediate]
 *   linear attention: dt_raw, b_raw [Hv], qkv [C], z, y [Hv*Dv], out, x_resid [hidden],
 *                     gate_act, up_act [intermediate]
 * The steps fused inside the kernel store plain bf16 values, and only while
 * qwen35_debug_stage_dump is on (the page's intra_dump names): x_norm, x_norm2
 * [hidden] (both kinds), qkv_smooth [C] and y_norm [Hv*Dv] (linear attention). */
QWEN35_API size_t qwen35_debug_scratch_offset(const qwen35_config* cfg, int layer_kind, const char* name);
QWEN35_API size_t qwen35_debug_stack_scratch_offset(const qwen35_config* cfg, const char* name);

/* Debug: while on (nonzero), the forwards launched after this call also store the
 * fused steps' values named above (x_norm, x_norm2, qkv_smooth, y_norm). Off by
 * default; not thread-safe. */
QWEN35_API int qwen35_debug_stage_dump(int on);

/* Debug: every bounded wait inside the kernels of the forwards launched after this
 * call gives up after limit_ns nanoseconds (0 restores the default of 1 s),
 * records QWEN35_ERR_DEVICE_TIMEOUT in the status word and lets the kernel run to
 * its end (its results are then meaningless). Copies into shared memory are always
 * waited for at least 1 s before a CTA exits. Not thread-safe; for tests. */
QWEN35_API int qwen35_debug_set_wait_limit(unsigned long long limit_ns);

/* Debug: with a non-null device pointer d_flag (4-byte aligned), the forwards
 * launched after this call run as usual, then thread 0 of every CTA waits (bounded
 * by the wait limit) for *d_flag to become nonzero before the kernel exits; a flag
 * that nothing sets makes that wait run out (QWEN35_ERR_DEVICE_TIMEOUT in the
 * status word) while the forward's results stay valid. NULL turns it off. Not
 * thread-safe; for tests. */
QWEN35_API int qwen35_debug_wait_probe(const uint32_t* d_flag);

/* Debug timeline of the forwards launched after this call (until it is called
 * again with NULL, 0): each CTA c (one per SM) writes, for phase f of a launch,
 * globaltimer readings (ns) at d_trace[(c * max_phases + f) * 16 + k]: k = 0
 * when it is done with the phase before, 1 when it enters the phase, 2 when
 * it finishes the phase; projection phases also write 3 when the phase's input
 * vector is formed and quantised, 4 and 5 when the first and the last of the
 * CTA's weight tiles is in shared memory, 6 when its rows are done; phases
 * that stream tiles write 7 when the first is requested; 8..12 mark steps inside
 * a projection phase (input loads landed, input stored, row loop entered, tile
 * loop entered, rows reduced). Entries a
 * phase does not write keep their contents. A phase is one step of a layer (6
 * per full-attention layer, 5 per linear-attention layer). d_trace is a device
 * buffer of #SMs * max_phases * 16 entries. Not thread-safe; for profiling. */
QWEN35_API int qwen35_debug_trace(unsigned long long* d_trace, uint32_t max_phases);

/* Dequantised weights of `w`, fp32 [n][k], each element fmaf(scale, code, bias) rounded
 * once: a check of the code/scale/bias indexing the GEMV uses. */
QWEN35_API int qwen35_dequant(const qwen35_qweight* w, float* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QWEN35_DECODE_H */
