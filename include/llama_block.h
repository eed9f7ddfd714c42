/*
 * llama_block.h -- C ABI of the GB300 (sm_103a) Llama pre-norm decoder block.
 *
 * Operation (one block, "Full Llama 3 transformer block", How it works):
 *     h = x + Attn(RMSNorm_1(x)),   y = h + FFN(RMSNorm_2(h))
 *   RMSNorm(x) = x / sqrt(mean(x^2) + norm_eps) * g        ("The Evolving Transformer 04 · LLaMA", §03)
 *   Attn: q = u Wq^T, k = u Wk^T, v = u Wv^T (no bias); RoPE rotates interleaved
 *         pairs (2i, 2i+1) of q and k by angle p * rope_theta^(-2i/d_head) at
 *         absolute position p = start_pos + s (§02 RoPE; "Mini Llama 2
 *         Implementation", Rotary positional embeddings); rotated k and raw v
 *         are written into the KV cache at positions [start_pos, start_pos + S);
 *         query head h attends to KV head h / (n_heads / n_kv_heads) over cache
 *         positions j <= start_pos + s with softmax(q.k / sqrt(d_head)) (§05 GQA);
 *         o is projected by Wo.
 *   FFN:  W_down(SiLU(W_gate v) * (W_up v))                 (§04 SwiGLU; How it works: W1, W3, W2)
 *
 * Conventions for every entry point below:
 *   - All tensor pointers are DEVICE pointers unless the name says _host.
 *   - Weights use nn.Linear layout [out_features, in_features], row-major.
 *   - Activations are token-major: x[b][s][d_model], row-major, contiguous.
 *   - dtype LLAMA_BF16: bf16 storage, fp32 accumulation; LLAMA_F32: fp32 throughout.
 *   - Functions that take a stream only ENQUEUE work on it (no host sync) and
 *     return after validation; a non-OK status means nothing was enqueued.
 *   - Every pointer must be 16-byte aligned (LLAMA_ERR_ALIGN otherwise).
 *   - Errors are returned, never raised or aborted on; llama_status_string()
 *     names them.  Kernels never trap: a device-side wait that exceeds its
 *     budget, or an out-of-range token id, sets the handle's device status
 *     word, read with llama_block_device_status() / llama_stack_device_status().
 */
#ifndef LLAMA_BLOCK_H
#define LLAMA_BLOCK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (CUstream) handle; NULL means the legacy default stream. */
typedef struct CUstream_st *llama_stream;

typedef enum {
    LLAMA_OK = 0,
    LLAMA_ERR_INVALID_ARG = 1,   /* null pointer, bad enum, non-positive size */
    LLAMA_ERR_SHAPE = 2,         /* d_model % n_heads, n_heads % n_kv_heads, odd d_head ... */
    LLAMA_ERR_ALIGN = 3,         /* a pointer is not 16-byte aligned */
    LLAMA_ERR_RANGE = 4,         /* start_pos + S beyond the cache / table, B beyond max_batch, T beyond max_tokens */
    LLAMA_ERR_UNSUPPORTED = 5,   /* valid Llama shape this build has no kernel for */
    LLAMA_ERR_OOM = 6,           /* device allocation failed in a create call */
    LLAMA_ERR_CUDA = 7,          /* a CUDA runtime/driver call failed */
    LLAMA_ERR_DEVICE_TIMEOUT = 8 /* a kernel's bounded wait ran out (see llama_block_device_status) */
} llama_status;

typedef enum { LLAMA_F32 = 0, LLAMA_BF16 = 1 } llama_dtype;

/* Which components of a head RoPE rotates together ("The Evolving Transformer
 * 04 · LLaMA", §02 RoPE and "Mini Llama 2 Implementation": interleaved pairs
 * (2i, 2i+1); "From GPT-2 to Llama: four changes and the reason for each",
 * Positions become a rotation: halves, pair i = (i, i + d_head/2), the
 * rotate_half form).  Pair i turns at the same frequency in both layouts. */
typedef enum { LLAMA_ROPE_INTERLEAVED = 0, LLAMA_ROPE_HALVES = 1 } llama_rope_layout;

/* Fields follow LlamaConfig / ModelArgs ("The Evolving Transformer 04 · LLaMA",
 * §00 Config; "Full Llama 3 transformer block", How it works).  d_head is
 * derived as d_model / n_heads.  max_seq_len bounds start_pos + S and sizes the
 * RoPE table.  Requirements: d_model % n_heads == 0, n_heads % n_kv_heads == 0,
 * d_head even and in {16, 32, 64, 128}, d_model and d_ff multiples of 8 (bf16)
 * or 4 (fp32), norm_eps >= 0, rope_theta > 0. */
typedef struct {
    int32_t d_model;
    int32_t n_heads;
    int32_t n_kv_heads;
    int32_t d_ff;
    int32_t max_seq_len;
    float norm_eps;
    float rope_theta;
    int32_t dtype; /* llama_dtype */
    /* RoPE variants ("From GPT-2 to Llama: four changes and the reason for
     * each", Positions become a rotation).  Zero-initialised fields give the
     * interleaved layout without scaling. */
    int32_t rope_layout;           /* llama_rope_layout */
    /* Llama 3.1 frequency stretch, applied when rope_scaling_factor > 1: with
     * wavelength lam_i = 2 pi / f_i and L = rope_original_max_pos, pairs with
     * lam_i < L / rope_high_freq_factor keep f_i, pairs with lam_i >
     * L / rope_low_freq_factor turn at f_i / rope_scaling_factor, and in
     * between f_i is blended as (1 - w) f_i / factor + w f_i with
     * w = (L / lam_i - low) / (high - low).  Requires 0 < low < high and L > 0. */
    float rope_scaling_factor;
    float rope_low_freq_factor;
    float rope_high_freq_factor;
    int32_t rope_original_max_pos;
    /* Mixture-of-experts feed-forward ("Llama 4 From Scratch", MoE; "From
     * GPT-2 to Llama: four changes and the reason for each", The feed-forward
     * grows a gate).  n_experts = 0: the dense SwiGLU of width d_ff.
     * n_experts > 0 (bf16 only): v = RMSNorm(h); router logits l = v W_router^T;
     * each token takes the top_k experts of largest logit (the lowest id among
     * equal logits) with weights softmax(l over the chosen experts); the
     * feed-forward output is sum_j w_j SwiGLU_{e_j}(v) (each expert of width
     * d_ff), plus SwiGLU_shared(v) of width d_ff_shared when d_ff_shared > 0.
     * Requires n_experts <= 256, 1 <= top_k <= min(n_experts, 32), d_model % 64
     * == 0, d_ff % 32 == 0, d_ff_shared % 32 == 0. */
    int32_t n_experts;
    int32_t top_k;
    int32_t d_ff_shared;
} llama_config;

/* Device pointers to one block's parameters, dtype = config.dtype.
 * attn_norm, ffn_norm: [d_model]; wq: [n_heads*d_head, d_model];
 * wk, wv: [n_kv_heads*d_head, d_model]; wo: [d_model, n_heads*d_head];
 * w_gate, w_up: [d_ff, d_model]; w_down: [d_model, d_ff].  No biases.
 * Mixture-of-experts blocks (n_experts > 0): w_gate, w_up: [n_experts][d_ff]
 * [d_model] and w_down: [n_experts][d_model][d_ff], one slice per expert;
 * router: [n_experts, d_model]; shared_gate, shared_up: [d_ff_shared, d_model]
 * and shared_down: [d_model, d_ff_shared] when d_ff_shared > 0.  The last four
 * are ignored (may be NULL) for dense blocks. */
typedef struct {
    const void *attn_norm, *wq, *wk, *wv, *wo, *ffn_norm, *w_gate, *w_up, *w_down;
    const void *router, *shared_gate, *shared_up, *shared_down;
} llama_block_weights;

/* Caller-owned KV cache of one layer: k and v are each
 * [max_batch][n_kv_heads][max_seq_len][d_head], dtype = config.dtype.  K is
 * stored after RoPE, V as projected.  Sequence b of a call uses row b.  A
 * forward call writes exactly positions [start_pos, start_pos + S) of rows
 * [0, B) and leaves every other element bit-for-bit unchanged. */
typedef struct {
    void *k;
    void *v;
    int32_t max_batch;
    int32_t max_seq_len;
} llama_kv_cache;

typedef struct llama_block llama_block;
typedef struct llama_stack llama_stack;

/* Validate cfg, copy/repack the weights into library-owned device memory (the
 * caller may free its copies afterwards) and reserve workspace for up to
 * max_tokens = B*S tokens per forward call.  Synchronous.  On error *out is
 * NULL and nothing stays allocated. */
llama_status llama_block_create(const llama_config *cfg, const llama_block_weights *w,
                                int32_t max_tokens, llama_block **out);

/* One block forward over x [B][S][d_model] -> y (same shape; y may alias x),
 * positions start_pos .. start_pos + S - 1 of each sequence, reading and
 * writing kv.  Requirements: 1 <= B <= kv->max_batch, S >= 1, B*S <= max_tokens,
 * 0 <= start_pos, start_pos + S <= min(cfg.max_seq_len, kv->max_seq_len).
 * Asynchronous on stream.  Calls on one llama_block must not overlap in time
 * (they share its workspace). */
llama_status llama_block_forward(llama_block *blk, const void *x, void *y, int32_t B, int32_t S,
                                 int32_t start_pos, const llama_kv_cache *kv, llama_stream stream);

/* Same as llama_block_forward but x_host / y_host are HOST buffers (pinned
 * memory recommended): copies x in, runs the block, copies y out, all on
 * stream; returns after enqueueing (synchronise the stream before reading
 * y_host).  The KV cache stays on the device. */
llama_status llama_block_forward_host(llama_block *blk, const void *x_host, void *y_host, int32_t B,
                                      int32_t S, int32_t start_pos, const llama_kv_cache *kv,
                                      llama_stream stream);

/* Routing of the most recent llama_block_forward of a mixture-of-experts block
 * (tracing, and for checking a forward against another implementation):
 * copies, on stream, ids int32 [B*S][top_k] (expert ids, in the order the
 * router chose them) and weights fp32 [B*S][top_k] into the caller's device
 * buffers.  LLAMA_ERR_INVALID_ARG for a dense block or before any forward. */
llama_status llama_block_moe_routing(llama_block *blk, int32_t *ids, float *weights, llama_stream stream);

void llama_block_destroy(llama_block *blk);

/* Full stack ("The Evolving Transformer 04 · LLaMA", §01 Embeddings, §07
 * Assemble): token embedding gather (no position table), n_layers blocks,
 * final RMSNorm, untied LM head.  embed: [vocab][d_model]; layers: array of
 * n_layers weight sets; final_norm: [d_model]; lm_head: [vocab][d_model]; all
 * device pointers of cfg.dtype, copied at create. */
llama_status llama_stack_create(const llama_config *cfg, int32_t n_layers, int32_t vocab,
                                const void *embed, const llama_block_weights *layers,
                                const void *final_norm, const void *lm_head, int32_t max_tokens,
                                llama_stack **out);

/* tokens: int32 [B][S] in [0, vocab) (device); kv: array of n_layers caches;
 * logits: fp32 [B][S][vocab] (device).  Same range rules as the block. */
llama_status llama_stack_forward(llama_stack *stk, const int32_t *tokens, int32_t B, int32_t S,
                                 int32_t start_pos, const llama_kv_cache *kv, float *logits,
                                 llama_stream stream);

/* Greedy decoding ("Full Llama 3 transformer block", How it works: the prompt
 * fills the cache at start_pos, then one new token per step at the next
 * position; "The Evolving Transformer 04 · LLaMA", §07 Assemble: the last
 * position's logits choose the next token).
 *   prompt     int32 [B][S_prompt] in [0, vocab) (device), run at start_pos;
 *   n_new      tokens to choose; each is the arg-max of the logits of the
 *              previous position (lowest id among equal maxima) and, except
 *              the last, is run as a one-token step at the next position;
 *   out_tokens int32 [B][n_new] (device), the chosen ids;
 *   logits     fp32 [B][vocab] (device), scratch; holds the logits that chose
 *              out_tokens[:, n_new - 1] on return;
 *   kv         n_layers caches; positions start_pos .. start_pos + S_prompt +
 *              n_new - 2 are written.
 * Range: B * S_prompt <= max_tokens, B <= kv.max_batch and start_pos +
 * S_prompt + n_new - 1 <= min(cfg.max_seq_len, kv.max_seq_len), else
 * LLAMA_ERR_RANGE.  Enqueues the whole loop on stream (no host sync): per
 * token the embedding gather, n_layers blocks, the final norm, the LM head and
 * the arg-max. */
llama_status llama_stack_generate(llama_stack *stk, const int32_t *prompt, int32_t B, int32_t S_prompt,
                                  int32_t start_pos, int32_t n_new, const llama_kv_cache *kv,
                                  int32_t *out_tokens, float *logits, llama_stream stream);

void llama_stack_destroy(llama_stack *stk);

/* Bytes of one layer's K plus V cache for max_batch x max_seq_len positions:
 * 2 * max_batch * n_kv_heads * max_seq_len * d_head * sizeof(dtype) ("Llama 4
 * From Scratch", Worked example: 2 x KV heads x head width per token).
 * Returns 0 for an invalid config. */
size_t llama_kv_cache_bytes(const llama_config *cfg, int32_t max_batch, int32_t max_seq_len);

/* SwiGLU inner width rule ("Full Llama 3 transformer block", How it works):
 * 4*d_model -> floor(2/3) -> floor(x ffn_dim_multiplier) when the multiplier
 * is > 0 -> round up to a multiple of multiple_of.  Returns -1 on bad input. */
int32_t llama_ffn_hidden_dim(int32_t d_model, int32_t multiple_of, float ffn_dim_multiplier);

const char *llama_status_string(llama_status s);

/* Text of the last CUDA error a call of this library returned LLAMA_ERR_CUDA
 * for, in the calling host thread ("no error" when none).  The pointer stays
 * valid until the next failing call in the same thread. */
const char *llama_last_cuda_error(void);

/* Number of CUDA kernels this library has launched since it was loaded, all
 * threads and handles together (tracing).  A launch captured into a CUDA graph
 * counts once, at capture; graph replays do not count.  Memsets are not kernels
 * of this library and are not counted. */
unsigned long long llama_kernel_launch_count(void);

/* Per-step timing of llama_block_forward (tracing).  When enabled, every
 * forward call records a CUDA event pair on its stream around each step's
 * kernel launch, for up to max_forwards calls (events are created here;
 * synchronous).  llama_block_profile_read synchronises the device, writes for
 * each step s in [0, LLAMA_PROFILE_STEPS) the number of forwards in which the
 * step launched a kernel of its own and the total milliseconds of those, then
 * clears the record; a step fused into another step's kernel (RoPE + KV write
 * in the QKV epilogue, ffn_norm in the O and gate/up epilogues) reads 0
 * launches.  Steps: 0 attention_norm,
 * 1 QKV projection, 2 RoPE + KV write, 3 attention, 4 O projection + residual,
 * 5 ffn_norm, 6 gate/up + SwiGLU, 7 down projection + residual. */
#define LLAMA_PROFILE_STEPS 8
llama_status llama_block_profile_enable(llama_block *blk, int32_t max_forwards);
llama_status llama_block_profile_disable(llama_block *blk);
llama_status llama_block_profile_read(llama_block *blk, int32_t *launches, float *total_ms);
const char *llama_profile_step_name(int32_t step);

/* How decode steps run ("Full Llama 3 transformer block", How it works: each
 * step feeds one new token per sequence through the block against the cache).
 * Applies to forwards with S == 1 of dense bf16 blocks whose d_head is 128;
 * every other forward always runs as one kernel per step.
 *   LLAMA_DECODE_KERNELS (default): one kernel per step of the block, each a
 *     programmatic dependent of the previous one;
 *   LLAMA_DECODE_FUSED: the whole block as one cooperative kernel (one CTA per
 *     SM) whose phases -- the same steps with the same tile plans -- are
 *     separated by grid-wide barriers.  Results equal the default's up to the
 *     order of fp32 reductions.  Fused forwards are not profiled.
 * Returns LLAMA_ERR_UNSUPPORTED (mode unchanged) when the device cannot run the
 * fused kernel, LLAMA_ERR_INVALID_ARG for an unknown mode.  Not thread-safe
 * against forwards of the same handle in flight on another host thread. */
typedef enum { LLAMA_DECODE_KERNELS = 0, LLAMA_DECODE_FUSED = 1 } llama_decode_mode;
llama_status llama_block_set_decode_mode(llama_block *blk, int32_t mode);
llama_status llama_stack_set_decode_mode(llama_stack *stk, int32_t mode);

/* Read and clear the handle's device status word.  Synchronises the device the
 * handle lives on.  Returns LLAMA_OK when no kernel reported a problem since
 * the last read, LLAMA_ERR_DEVICE_TIMEOUT when a bounded wait ran out,
 * LLAMA_ERR_RANGE when a token id was outside [0, vocab) (its embedding row
 * was written as zeros), LLAMA_ERR_CUDA when the read itself failed. */
llama_status llama_block_device_status(llama_block *blk);
llama_status llama_stack_device_status(llama_stack *stk);

/* Bound, in SM clock cycles, on every wait of this handle's kernels that gives
 * up (mbarrier waits of the tensor-core kernels, the fused decode kernel's
 * phase barriers, the split-KV decode kernel's stage waits); 0 restores the
 * default, about 4e9 cycles (2 s at 2 GHz), which no legitimate wait reaches.
 * A wait that runs out records LLAMA_ERR_DEVICE_TIMEOUT in the status word
 * (llama_block_device_status), makes the kernel's other roles give up too, and
 * the kernel returns once the copies and MMAs it had issued have completed --
 * those waits keep the default bound -- and its tensor memory is freed; the
 * outputs of that forward are undefined, the context stays usable, and
 * reading the status resets the handle's scratch for the next forward.  This
 * is a fault-injection and diagnosis knob (a short budget makes ordinary
 * waits give up); the library itself never sets it.  Synchronises the
 * device; do not call it while a forward of the handle is in flight.
 * LLAMA_ERR_INVALID_ARG for a null handle or a negative budget.
 * The pages have no counterpart: it serves the bounded-wait failure
 * detection of the kernels. */
llama_status llama_block_set_wait_budget(llama_block *blk, int64_t cycles);
llama_status llama_stack_set_wait_budget(llama_stack *stk, int64_t cycles);

#ifdef __cplusplus
}
#endif
#endif /* LLAMA_BLOCK_H */
