/*
 * switch_moe.h -- C ABI of libswitchmoe.so, the forward pass of a Switch-style
 * top-1 Mixture-of-Experts FFN layer on one NVIDIA B300 (sm_103a).
 *
 * The layer, per token x_t (a row of x):
 *   1. router logits  l_t = W_g x_t (+ b_g)                      [fp32]
 *   2. score = softmax(l_t); expert_id = argmax; gate = score[expert_id]
 *   3. capacity C = ceil(capacity_factor * T / N)
 *   4. slot of the token in its expert's buffer; tokens past C are dropped
 *   5. dispatch x_t into buffer [N, C, d_model]
 *   6. expert FFN: o = W2_e relu(W1_e x_t)
 *   7. combine:  y_t = (gate_multiply ? gate : 1) * o, or 0 if dropped,
 *                plus the shared expert's FFN of x_t when there is one
 *   8. L_aux = N * sum_i f_i * P_i
 *
 * Sources (page title, then section / equation / figure):
 *   [TOP1]   "Top-1 路由 (Top-1 Routing)", compassingai.com: core mechanism
 *            steps 1-3 (steps 1, 2, 6, 7 above), load-balancing section
 *            (step 8), Token Dropping section (steps 3, 4), key-parameter
 *            section (two-layer FFN without bias).
 *   [SWITCH] Switch Transformer walk-through, personwebsite.pages.dev/
 *            moe-switch: Switch layer (the gate as multiplier, Eq. 2),
 *            expert-capacity section (dropped tokens skip the expert and
 *            continue through the residual), load-balancing loss (Eq. 4),
 *            selective precision (the router computes in float32).
 *   [CAP]    "MoE 专家容量因子与 Token 丢弃", wiblog.cn: capacity formula and
 *            the fixed-shape per-expert buffer (section on where capacity
 *            comes from), overflow by routing-weight priority (section on
 *            overflow handling; flowchart nodes D -> F).
 *   [CMP]    "Which Routing Does Each MoE Model Use?" (MarkTechPost digest),
 *            routing table: top-1 over 128 experts plus one shared expert.
 *
 * Conventions for every entry point
 *   - Device pointers unless a name says "host".  The caller allocates and
 *     owns every buffer (inputs, outputs, workspace); the library never
 *     allocates, frees or synchronises inside a compute call, so calls can
 *     be captured in a CUDA graph.  Work is enqueued on `stream` (NULL =
 *     legacy default stream) and runs asynchronously.
 *   - Matrices are dense row-major.  x [T, d_model]; W_g [N, d_model] fp32;
 *     b_g [N] fp32 or NULL; W1 [N, d_ff, d_model]; W2 [N, d_model, d_ff];
 *     W1s [d_ff, d_model] and W2s [d_model, d_ff] (shared expert) or NULL;
 *     y [T, d_model] fp32.  x, W1, W2, W1s, W2s have the element type
 *     `dtype` (fp32 or bf16).
 *   - Alignment: x, W1, W2, W1s, W2s, y, logits and the workspace must be
 *     16-byte aligned (the workspace 256-byte aligned); int/float vectors
 *     4-byte aligned.
 *   - Return value: SWITCH_MOE_OK (0) or a negative SWITCH_MOE_ERR_* code.
 *     Argument errors are found on the host before anything is enqueued.
 *     A device-side failure (a bounded wait that expired) is recorded in a
 *     per-device status word and reported by switch_moe_sync_status().
 *   - Inputs must be finite; NaN/Inf inputs give unspecified outputs.
 */
#ifndef SWITCH_MOE_H
#define SWITCH_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (both are pointers to the same opaque CUDA type). */
typedef struct CUstream_st* switch_moe_stream_t;

enum switch_moe_status {
  SWITCH_MOE_OK = 0,
  SWITCH_MOE_ERR_INVALID_ARG = -1,         /* sizes <= 0, bad enum, NULL pointer, cf not finite > 0 */
  SWITCH_MOE_ERR_ALIGNMENT = -2,           /* a pointer breaks the alignment rules above */
  SWITCH_MOE_ERR_WORKSPACE_TOO_SMALL = -3, /* workspace_bytes < switch_moe_workspace_bytes() */
  SWITCH_MOE_ERR_UNSUPPORTED = -4,         /* shape outside the supported range (see below) */
  SWITCH_MOE_ERR_CUDA = -5,                /* a CUDA runtime call or kernel launch failed */
  SWITCH_MOE_ERR_DEVICE_TIMEOUT = -6,      /* a device-side bounded wait expired */
  SWITCH_MOE_ERR_NO_DEVICE = -7            /* no usable sm_103 device is current */
};

enum switch_moe_priority {
  SWITCH_MOE_TOKEN_ORDER = 0,   /* earlier tokens fill an expert first */
  SWITCH_MOE_GATE_PRIORITY = 1  /* higher gate first, ties by lower token index [CAP] */
};

enum switch_moe_dtype {
  SWITCH_MOE_F32 = 0,   /* x, W1, W2 (and W1s, W2s) fp32; exact fp32 FFN */
  SWITCH_MOE_BF16 = 1   /* bf16 operands, fp32 accumulation on tcgen05 tensor cores */
};

/* Layer shape and options.  Supported range:
 *   1 <= N <= 1024; d_model, d_ff >= 8 and multiples of 8;
 *   T >= 0 (T == 0 is a no-op that zeroes expert_counts and aux_loss);
 *   capacity C >= 1; gate-priority mode needs min(C, T) <= 16384. */
typedef struct switch_moe_params {
  int64_t T;                /* tokens in the batch */
  int64_t d_model;
  int64_t d_ff;
  int64_t N;                /* routed experts */
  double capacity_factor;   /* cf > 0 */
  int32_t priority_mode;    /* enum switch_moe_priority */
  int32_t gate_multiply;    /* 1: y = gate * E(x) ([SWITCH] Eq. 2); 0: y = E(x) ([TOP1] step 3) */
  int32_t dtype;            /* enum switch_moe_dtype */
  int32_t has_shared;       /* 1: add an always-on shared expert W1s/W2s ([CMP]) */
  /* Expanded Drop ([CAP] inference section): 0 or 1 = off (plain top-1);
   * k in 2..4 = each token's candidate set is its first k experts by logit
   * (lowest index first on ties); tokens the top-1 pass drops take, in token
   * order, the next free slot of their 2nd, then 3rd, ... candidate.  A
   * re-routed token runs on that expert with that expert's probability as
   * its gate; expert_id / gate / slot report the expert that runs it.
   * expert_counts and aux_loss keep the router's top-1 choices.  Token-order
   * priority only (SWITCH_MOE_ERR_UNSUPPORTED otherwise); k <= N. */
  int32_t expand;
  /* Experts per token: 0 or 1 = top-1 (Switch); 2 = top-2 token choice
   * ([TOP1] industry-position and comparison sections: GShard and Mixtral
   * send every token to two experts and merge the outputs with weights;
   * [SWITCH] Switch-layer section: the top-k layer's output is the
   * gate-weighted sum over the chosen set).  The chosen pair is the two
   * highest logits, lowest index first on ties; choice 0 is the top-1
   * expert.  Capacity is the same C = ceil(cf * T / N) (pass a larger cf to
   * make room for both choices).  Slots: every token's choice 0 in token
   * order first (the top-1 assignment), then every token's choice 1 in
   * token order after the slots its expert already holds; a choice is kept
   * iff its slot < C.  y[t] = sum over the kept choices of g * E(x_t) (+ the
   * shared expert); a dropped choice adds nothing.  With top_k == 2 the
   * per-token outputs expert_id, gate, slot and drop_mask are [T, 2]
   * (row-major, choice fastest); expert_counts and aux_loss count choice 0
   * (the router's top-1).  Token-order priority, N >= 2 and expand <= 1
   * only (SWITCH_MOE_ERR_UNSUPPORTED otherwise).  The two adds into a y row
   * are atomic: with a shared expert (three terms) their order, and so the
   * last bit of y, can differ between runs. */
  int32_t top_k;
  /* top_k == 2 only (SWITCH_MOE_ERR_INVALID_ARG otherwise): 0 = the gates are
   * the chosen experts' softmax probabilities over all N; 1 = softmax over
   * the two chosen logits, p_e / (p_e0 + p_e1) ([CMP] routing table,
   * Mixtral: softmax over the top-k). */
  int32_t renormalize;
  /* 1 = expert-choice routing, used only by switch_moe_forward_expert_choice()
   * and switch_moe_route_expert_choice() (the token-choice entry points
   * return SWITCH_MOE_ERR_INVALID_ARG for it); 0 otherwise.  Needs top_k <= 1,
   * expand <= 1 and min(C, T) <= 16384 (SWITCH_MOE_ERR_UNSUPPORTED). */
  int32_t expert_choice;
} switch_moe_params;

/* Expert capacity C = ceil(cf * T / N), evaluated in double as (cf*T)/N.
 * [TOP1] Token Dropping section; [CAP] capacity formula.  The pages give no
 * rounding; ceil is this library's reading.  Returns C >= 1, or
 * SWITCH_MOE_ERR_INVALID_ARG when T < 1, N < 1, cf is not finite > 0 or C
 * would not fit in 31 bits.  Pure host function. */
int64_t switch_moe_capacity(int64_t T, int64_t N, double capacity_factor);

/* Bytes of device workspace switch_moe_forward() needs for `p`, written to
 * *bytes.  Returns an error code for an invalid or unsupported `p`.  Host
 * only; no device is touched. */
int switch_moe_workspace_bytes(const switch_moe_params* p, size_t* bytes);

/* The whole layer forward (steps 1-8 above) on `stream`.
 * Inputs:  x, W_g, b_g (nullable), W1, W2, W1s/W2s (only read when
 *          p->has_shared; may be NULL otherwise).
 * Outputs: y             [T, d_model] fp32: the MoE branch; the caller adds
 *                        the residual ([TOP1] Transformer-block figure:
 *                        "LayerNorm + Residual" follows the layer), so a
 *                        dropped token's x + y is x (plus the shared expert).
 *          expert_id     [T] int32, argmax of the fp32 logits, lowest index on ties
 *          gate          [T] fp32,  softmax probability of expert_id
 *          slot          [T] int32, position in the expert buffer, -1 if dropped
 *          drop_mask     [T] uint8, 1 if dropped
 *          expert_counts [N] int32, tokens routed to each expert before capacity
 *          aux_loss      [1] fp32,  N * sum_i f_i P_i, f_i = counts_i / T,
 *                        P_i = mean_t score_t[i] (not multiplied by alpha)
 * workspace: device scratch of at least switch_moe_workspace_bytes(p); its
 *          contents on entry do not matter; it must not be shared by two
 *          calls that may run at the same time. */
int switch_moe_forward(const switch_moe_params* p,
                       const void* x, const float* W_g, const float* b_g,
                       const void* W1, const void* W2,
                       const void* W1s, const void* W2s,
                       float* y, int32_t* expert_id, float* gate, int32_t* slot,
                       uint8_t* drop_mask, int32_t* expert_counts, float* aux_loss,
                       void* workspace, size_t workspace_bytes,
                       switch_moe_stream_t stream);

/* Steps 2-4 and 8 on given fp32 logits [T, N] (row-major): softmax, argmax,
 * gate, capacity, slot assignment, drop mask, counts and L_aux, exactly as
 * switch_moe_forward() takes them from its own logits.  Uses p->T, p->N,
 * p->capacity_factor and p->priority_mode; the other fields are ignored
 * (d_model and d_ff may be 0).  Workspace: switch_moe_workspace_bytes() of a
 * params struct with the same T and N and d_model = d_ff = 8. */
int switch_moe_route_from_logits(const switch_moe_params* p, const float* logits,
                                 int32_t* expert_id, float* gate, int32_t* slot,
                                 uint8_t* drop_mask, int32_t* expert_counts,
                                 float* aux_loss, void* workspace,
                                 size_t workspace_bytes, switch_moe_stream_t stream);

/* switch_moe_route_from_logits() for callers that cannot allocate device
 * memory when they route: for example a server that gave all of its device
 * memory to a pool at start-up and allows no cudaMalloc afterwards, or a
 * runtime with a memory budget fixed before the first request.  There is no
 * workspace argument; the scratch lives in a static device array of about
 * 1.2 MiB that every GPU loading the library holds until the process exits.
 * (The pages have no counterpart to this entry point; it is an interface
 * convenience of this library.)
 *   Limits: p->T <= 16384 tokens and p->N <= 256 experts; larger sizes
 *   return SWITCH_MOE_ERR_UNSUPPORTED and enqueue nothing.
 *   The first call on a device looks up the array's device address (once
 *   per device, with that device current); make that first call before any
 *   stream capture.
 *   Every call uses the same array: calls that overlap on the GPU (other
 *   streams, other host threads on the same device) race and must not be
 *   issued; calls on one stream are ordered and safe.  Nothing left from an
 *   earlier call is read.
 *   Outputs and their meaning are those of switch_moe_route_from_logits(). */
int switch_moe_route_from_logits_noalloc(const switch_moe_params* p, const float* logits,
                                         int32_t* expert_id, float* gate, int32_t* slot,
                                         uint8_t* drop_mask, int32_t* expert_counts,
                                         float* aux_loss, switch_moe_stream_t stream);

/* Expert-choice routing ([TOP1] routing-paradigm table: each expert selects
 * its top-K tokens; milestone table: Expert Choice Routing, Zhou et al.;
 * comparison table: a token can be taken by several experts or by none).
 * p->expert_choice must be 1.  The scores are the top-1 layer's router,
 * s[t, e] = softmax over the N experts of token t's fp32 logits.  Each
 * expert takes k = min(C, T) tokens, C = ceil(cf * T / N): those with the
 * highest s[:, e], the lower token index first among equal scores; slot =
 * rank.  y[t] = sum over the experts that took t of g * E_e(x_t), g = s[t, e]
 * (1 when gate_multiply is 0), plus the shared expert; 0 when no expert
 * took t.  (The pages print no formula for expert choice; this is the
 * plainest reading of the tables.)
 * Outputs: y                 [T, d_model] fp32
 *          chosen_token      [N, C] int32: expert e's tokens, best first; -1 past T
 *          chosen_gate       [N, C] fp32: their scores s[t, e]; 0 past T
 *          experts_per_token [T] int32: how many experts took each token
 *          expert_counts     [N] int32 and aux_loss [1]: the router's top-1
 *                            statistics (counts of argmax and L_aux, as in
 *                            switch_moe_forward; expert choice itself needs no
 *                            balancing loss)
 * The adds of several slots into a y row are atomic: their order, and so the
 * last bit of y, can differ between runs.  Workspace, alignment and errors as
 * for switch_moe_forward(). */
int switch_moe_forward_expert_choice(const switch_moe_params* p,
                                     const void* x, const float* W_g, const float* b_g,
                                     const void* W1, const void* W2,
                                     const void* W1s, const void* W2s,
                                     float* y, int32_t* chosen_token, float* chosen_gate,
                                     int32_t* experts_per_token, int32_t* expert_counts,
                                     float* aux_loss, void* workspace, size_t workspace_bytes,
                                     switch_moe_stream_t stream);

/* The routing of switch_moe_forward_expert_choice() on given fp32 logits
 * [T, N]: the same outputs without y.  Workspace: switch_moe_workspace_bytes()
 * of a params struct with the same T, N and cf, expert_choice = 1 and
 * d_model = d_ff = 8. */
int switch_moe_route_expert_choice(const switch_moe_params* p, const float* logits,
                                   int32_t* chosen_token, float* chosen_gate,
                                   int32_t* experts_per_token, int32_t* expert_counts,
                                   float* aux_loss, void* workspace, size_t workspace_bytes,
                                   switch_moe_stream_t stream);

/* Backward of the top-1 layer ([SWITCH] load-balancing section: the
 * auxiliary loss joins the training loss with a coefficient; [TOP1] core
 * mechanism steps 1-3 and load-balancing section): the gradients of
 * <dy, y> + aux_coef * L_aux with respect to x, W_g, b_g, W1, W2 (and W1s,
 * W2s), where y is switch_moe_forward()'s output for the same inputs.
 * Inputs: the forward's inputs (x, W_g, b_g, W1, W2, W1s, W2s; p as for the
 *         forward), its routing outputs expert_id, gate, slot [T] and
 *         expert_counts [N], and dy [T, d_model] fp32.
 * Outputs (fp32, row-major, the layouts of the forward's operands):
 *         dx [T, d_model]; dW_g [N, d_model]; db_g [N] (nullable: not
 *         computed); dW1 [N, d_ff, d_model]; dW2 [N, d_model, d_ff]; dW1s
 *         [d_ff, d_model], dW2s [d_model, d_ff] with a shared expert.
 * Readings: the routing decisions (argmax, capacity, slots) are piecewise
 * constant and get no gradient, so f_i is constant and dL_aux/dp[t, i] =
 * N f_i / T; the gate gets dy . E(x) when gate_multiply is set; ReLU'(0) = 0.
 * The forward's intermediates are recomputed in fp32 from the inputs (bf16
 * inputs widened exactly) on FFMA.  Top-1 only (expand, top_k and
 * expert_choice give SWITCH_MOE_ERR_UNSUPPORTED).  Workspace: at least
 * switch_moe_backward_workspace_bytes(p); alignment and errors as for
 * switch_moe_forward(). */
int switch_moe_backward_workspace_bytes(const switch_moe_params* p, size_t* bytes);
int switch_moe_backward(const switch_moe_params* p, const void* x, const float* W_g,
                        const float* b_g, const void* W1, const void* W2, const void* W1s,
                        const void* W2s, const int32_t* expert_id, const float* gate,
                        const int32_t* slot, const int32_t* expert_counts, const float* dy,
                        float aux_coef, float* dx, float* dW_g, float* db_g, float* dW1,
                        float* dW2, float* dW1s, float* dW2s, void* workspace,
                        size_t workspace_bytes, switch_moe_stream_t stream);

/* Step 1 alone: logits [T, N] fp32 = x W_g^T (+ b_g), computed by the same
 * device code that switch_moe_forward() fuses with steps 2-4, so feeding
 * these logits to switch_moe_route_from_logits() reproduces the forward
 * pass's routing bit for bit ([SWITCH] selective precision: fp32 router).
 * Uses p->T, p->d_model, p->N and p->dtype (the type of x).  workspace: at
 * least switch_moe_workspace_bytes() of a params struct with the same T,
 * d_model, N and dtype and d_ff = 8 (bf16 layers keep the split router
 * weights there). */
int switch_moe_router_logits(const switch_moe_params* p, const void* x,
                             const float* W_g, const float* b_g, float* logits,
                             void* workspace, size_t workspace_bytes,
                             switch_moe_stream_t stream);

/* switch_moe_forward() with HOST input and output buffers, for callers whose
 * activations live in host memory.  x_host [T, d_model] (dtype) is copied to
 * the device, the layer runs, and every output is copied back into the
 * *_host buffers, all enqueued on `stream` (pinned host memory makes the
 * copies asynchronous).  The host outputs are valid after the stream is
 * synchronised.  Weights stay device pointers.  Workspace: at least
 * switch_moe_hostio_workspace_bytes(p) (it also holds device copies of x
 * and of the outputs). */
int switch_moe_hostio_workspace_bytes(const switch_moe_params* p, size_t* bytes);
int switch_moe_forward_hostio(const switch_moe_params* p,
                              const void* x_host, const float* W_g, const float* b_g,
                              const void* W1, const void* W2,
                              const void* W1s, const void* W2s,
                              float* y_host, int32_t* expert_id_host, float* gate_host,
                              int32_t* slot_host, uint8_t* drop_mask_host,
                              int32_t* expert_counts_host, float* aux_loss_host,
                              void* workspace, size_t workspace_bytes,
                              switch_moe_stream_t stream);

/* Synchronises `stream`, then returns and clears the current device's status
 * word: SWITCH_MOE_OK, SWITCH_MOE_ERR_DEVICE_TIMEOUT if a kernel gave up a
 * bounded wait since the last call, or SWITCH_MOE_ERR_CUDA if the
 * synchronisation itself failed. */
int switch_moe_sync_status(switch_moe_stream_t stream);

/* Static, NUL-terminated description of a status code. */
const char* switch_moe_strerror(int code);

/* Benchmark aid.  With `events` pointing to SWITCH_MOE_NUM_PHASE_EVENTS
 * cudaEvent_t handles (created by the caller), every later
 * switch_moe_forward() / switch_moe_forward_hostio() call from this host
 * thread records them on its stream at the phase boundaries below, so
 * cudaEventElapsedTime between consecutive events times each kernel on the
 * stream it runs on.  events == NULL switches recording off.  Returns
 * SWITCH_MOE_ERR_INVALID_ARG when n != SWITCH_MOE_NUM_PHASE_EVENTS.
 *   0 start              1 after the router        2 after the scan (L_aux)
 *   3 after slots + dispatch
 *   4 after the shared-expert GEMMs (== 3 without one)
 *   5 after the routed experts' GEMM 1 (== 4 when one launch runs both layers)
 *   6 after the routed experts' GEMM 2
 *   7 after combine (== 6 when GEMM 2's epilogue combines) */
#define SWITCH_MOE_NUM_PHASE_EVENTS 8
int switch_moe_set_phase_events(void* const* events, int n);

/* Diagnostic: runs one kernel whose single bounded wait is on an mbarrier
 * that nothing ever arrives on, with a limit of `timeout_ns` (clamped to
 * [1 ms, 2 s]).  The wait gives up, the kernel records
 * SWITCH_MOE_ERR_DEVICE_TIMEOUT in the status word and exits normally, so
 * switch_moe_sync_status() then reports the timeout and clears it.  It
 * exercises the same wait routine every pipelined kernel of the library
 * uses, without faulting or hanging the device. */
int switch_moe_selftest_wait_timeout(uint64_t timeout_ns, switch_moe_stream_t stream);

/* Library version as major*10000 + minor*100 + patch. */
int switch_moe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SWITCH_MOE_H */
