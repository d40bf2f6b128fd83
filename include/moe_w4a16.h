/*
 * moe_w4a16.h -- C ABI of the W4A16 MoE expert layer for GB300 (sm_103a).
 *
 * The layer (per denoising step of a block-diffusion LM; model card
 * "srswti/axe-diffusion-ksl-xe", sections "what the model is" and "the kernels
 * we built"):
 *   1. route:   each of T tokens picks its top-k of E experts from fp32 router
 *               logits; the k selected logits are softmax-normalised;
 *   2. expert:  each (token, expert) pair runs the expert's gated-GELU FFN
 *               h = gelu(Wg x) * (Wu x),  y = Wd h,  with Wg|Wu|Wd stored as
 *               uint4 codes with an fp16 scale and a second fp16 value per
 *               group along the contraction dim -- by default asymmetric,
 *               w = (q - z) * s; affine w = q * s + b and symmetric
 *               w = (q - 8) * s are selectable (moe_w4a16_shape.format) --
 *               dequantised inside the GEMM ("the kernels we built": the GEMM
 *               reads packed nibbles and dequantises inline), in one of two
 *               reduction orders (moe_w4a16_shape.reduction);
 *   3. combine: out[t] = sum over router ranks r = 0..k-1, in rank order, of
 *               w[t][r] * y[t][r], in fp32 with no atomics ("the kernels we
 *               built": fixed-order combine instead of index_add_), optionally
 *               followed by an fp32 RMSNorm ("the kernels we built": fused
 *               RMSNorm).
 * Beside the layer, moe_w4a16_sample runs the per-step sampler of the
 * denoising loop (entropy, Gumbel-max token, acceptance of positions) in one
 * streaming pass over the vocabulary logits (see its section below).
 * The weight format follows the model card's "requirements" paragraph
 * (dg-w4a16-v1: two nibbles per byte; gate_up_proj grouped along the
 * contraction dim; down_proj grouped at 64 because its contraction dim, 704, is
 * not a multiple of 128).
 *
 * Conventions for every call:
 *   - Device pointers are allocated and owned by the caller; the library
 *     allocates nothing, never synchronises the host (except
 *     moe_w4a16_read_error), and launches only on the given stream
 *     (a cudaStream_t passed as void*, NULL = legacy default stream).
 *   - Shapes and pointers are validated on the host before anything is
 *     launched; on any status other than MOE_W4A16_OK nothing was launched
 *     and no output was written.  The library never reads device data to
 *     validate it: out-of-range device contents (e.g. an expert id >= E in a
 *     caller-built routing) are the caller's responsibility.
 *   - fp16 values travel as uint16_t bit patterns (IEEE binary16).
 *   - Every device pointer of the layer's calls must be 16-byte aligned (the
 *     sampler's rules are in its section).
 *   - Calls sharing one workspace must not overlap in time (same stream, or
 *     ordered by events); calls with separate workspaces are independent.
 *   - Results are bit-identical from run to run for the same inputs and shape:
 *     no floating-point atomics are used and every reduction has a fixed order.
 */
#ifndef MOE_W4A16_H
#define MOE_W4A16_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_W4A16_API __attribute__((visibility("default")))
#else
#define MOE_W4A16_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_W4A16_OK = 0,
  MOE_W4A16_ERR_NULL = 1,      /* a required pointer is NULL */
  MOE_W4A16_ERR_SHAPE = 2,     /* shape outside the supported set (see moe_w4a16_shape) */
  MOE_W4A16_ERR_ALIGN = 3,     /* a device pointer is not 16-byte aligned */
  MOE_W4A16_ERR_WORKSPACE = 4, /* workspace smaller than moe_w4a16_workspace_bytes() */
  MOE_W4A16_ERR_CUDA = 5,      /* a CUDA runtime call or kernel launch failed */
  MOE_W4A16_ERR_DEVICE = 6,    /* current device is not a compute capability 10.3 GPU */
  MOE_W4A16_ERR_TIMEOUT = 7,   /* a device-side wait ran out (reported by moe_w4a16_read_error) */
  MOE_W4A16_ERR_VALUE = 8      /* host data out of range (a code > 15, a scale or zero the kernels cannot hold) */
} moe_w4a16_status;

/* Layer shape.
 *   tokens        T >= 0 (T = 0 is an OK no-op)
 *   hidden        d, a multiple of 128
 *   inter         f (expert FFN width), a multiple of 64
 *   experts       E, 1..256
 *   top_k         k, 1..min(E, 8)
 *   group_gate_up g1 in {32, 64, 128}, dividing d: quantisation group of gate_up_proj along d
 *   group_down    g2 in {32, 64, 128}, dividing f: quantisation group of down_proj along f
 *   activation    0 = GELU tanh form 0.5a(1+tanh(sqrt(2/pi)(a+0.044715a^3))), 1 = GELU erf form
 *   reduction     order of the expert GEMMs' arithmetic (both give the layer within the same
 *                 tolerance, each bit-reproducible and independent of the other tokens):
 *                 0 = each weight dequantised to fp16, w = fp16((q - zr) s - fp16((z - zr) s)) with
 *                     zr the integer nearest z, and multiplied into fp32 accumulators in
 *                     contraction order;
 *                 1 = group-factorised, the int4 GEMM order of "ashhart/TensorFold pull 802"
 *                     (section "Contracts": partial sums per group, then the scale, then the
 *                     bias): per quantisation group the codes are multiplied as they are into
 *                     fp32 partial sums, then the group's scale is applied and its zero-point
 *                     term -s z sum(x) added, group after group.  More accurate (no weight is
 *                     rounded to fp16); work items of at most 16 tokens, so slower than 0 when
 *                     experts get more than ~8 tokens each
 *   format        weight format, one fp16 scale s and one fp16 second value per group
 *                 ("ashhart/TensorFold pull 802", "Summary": symmetric GPTQ 4/128 and MLX affine
 *                 4/64 checkpoints beside the model card's asymmetric uint4):
 *                 0 = asymmetric zero-point, w = (q - z) s, 0 <= z <= 16 (dg-w4a16-v1);
 *                 1 = affine bias (MLX), w = q s + b, |b| <= 1024 (the second value is b);
 *                 2 = symmetric (GPTQ), w = (q - 8) s (no second value: moe_w4a16_prepare
 *                     writes 8 and accepts zero == NULL)
 * T*k must not exceed 2^22. */
typedef struct {
  int32_t tokens, hidden, inter, experts, top_k, group_gate_up, group_down, activation, reduction, format;
} moe_w4a16_shape;

/* Expert weights of one layer, in the prepared layout written by
 * moe_w4a16_prepare (see there); device pointers, read only.
 *   gate_up  moe_w4a16_prepared_bytes(shape, MOE_W4A16_GATE_UP) bytes
 *   down     moe_w4a16_prepared_bytes(shape, MOE_W4A16_DOWN) bytes */
typedef struct {
  const uint8_t* gate_up;
  const uint8_t* down;
} moe_w4a16_weights;

/* Routing of one canvas, written by moe_w4a16_route, read by moe_w4a16_forward
 * (device pointers):
 *   topk_idx        int32 [T][k]   expert ids in router-rank order (rank 0 = largest logit)
 *   topk_w          fp32  [T][k]   softmax over the k selected logits
 *   expert_offsets  int32 [E+1]    pairs of expert e are pair_list[offsets[e] .. offsets[e+1])
 *   pair_list       int32 [T*k]    pair ids p = t*k + r grouped by expert, p ascending within an expert */
typedef struct {
  int32_t* topk_idx;
  float* topk_w;
  int32_t* expert_offsets;
  int32_t* pair_list;
} moe_w4a16_routing;

#define MOE_W4A16_GATE_UP 0
#define MOE_W4A16_DOWN 1

/* Bytes of device workspace that moe_w4a16_route and moe_w4a16_forward need for
 * this shape (0 on an invalid shape).  The workspace holds the intermediate
 * activations h (fp16 [T*k][f]), the token rows copied in expert order
 * (fp16 [T*k][d]), per-pair expert outputs (fp32 [T*k][d]) and routing scratch
 * (per-CTA expert counts, per-pair ranks) plus a small header (error word, work
 * counters), plus, for moe_w4a16_block, the normalised input u (fp16 [T][d]) and
 * the router logits (fp32 [T][E]).  It must be initialised once with
 * moe_w4a16_workspace_init before its first use; later calls leave it ready. */
MOE_W4A16_API size_t moe_w4a16_workspace_bytes(const moe_w4a16_shape* shape);

/* Clears the workspace header (error word and work counters) on `stream`. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* Routing (step 1): top-k, softmax over the selected logits, and the per-expert
 * pair lists.  Ties between equal logits go to the lower expert index (compared
 * as fp32 values, so -0 ties +0).  Logits must be finite; NaN or infinite
 * logits give unspecified (but in-bounds) routing.
 *   logits  fp32 [T][E], device, read only
 *   out     the four routing arrays, device, written */
MOE_W4A16_API moe_w4a16_status moe_w4a16_route(const moe_w4a16_shape* shape, const float* logits, const moe_w4a16_routing* out,
                                 void* workspace, size_t workspace_bytes, void* stream);

/* Expert FFNs and combine (steps 2 and 3).
 *   x           fp16 [T][d], device, read only
 *   routing     as written by moe_w4a16_route (read only)
 *   weights     prepared weights of this layer
 *   norm_gamma  fp32 [d] or NULL; when given, out = fp16(gamma * u / sqrt(mean(u^2) + norm_eps))
 *               with u the fp32 combine result; when NULL, out = fp16(u)
 *   out         fp16 [T][d], device, written; must not overlap x or the workspace
 * Rounding: fp16 results are rounded to nearest even. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_forward(const moe_w4a16_shape* shape, const uint16_t* x, const moe_w4a16_routing* routing,
                                   const moe_w4a16_weights* weights, const float* norm_gamma, float norm_eps,
                                   uint16_t* out, void* workspace, size_t workspace_bytes, void* stream);

/* The expert FFNs of moe_w4a16_forward without the combine: the gate_up and
 * down GEMMs of every (token, expert) pair in one persistent launch, in which a
 * down work item starts as soon as its expert's gate_up items have written
 * their h rows ([MC] "the kernels we built": one launch for all experts).
 * Leaves h and the per-pair rows y in the workspace for moe_w4a16_combine.
 * Same arguments and rules as moe_w4a16_forward. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_experts(const moe_w4a16_shape* shape, const uint16_t* x,
                                                 const moe_w4a16_routing* routing, const moe_w4a16_weights* weights,
                                                 void* workspace, size_t workspace_bytes, void* stream);

/* The steps of moe_w4a16_forward, callable one by one on the same stream in
 * this order (same arguments and rules as moe_w4a16_forward; e.g. to time each
 * step or to interleave other work); gate_up followed by down computes what
 * moe_w4a16_experts computes, in two launches:
 *   moe_w4a16_gate_up  expert gate_up GEMMs with the gated GELU folded into the
 *                      epilogue: h = gelu(Wg x) * (Wu x) for every (token, expert)
 *                      pair -> fp16 rows in the workspace, ordered by expert
 *   moe_w4a16_down     expert down GEMMs: y = Wd h -> fp32 rows in the workspace,
 *                      one per pair p = t*k + r
 *   moe_w4a16_combine  out[t] = fp16(sum_r w[t][r] y[t*k+r]) in rank order, with the
 *                      optional RMSNorm */
MOE_W4A16_API moe_w4a16_status moe_w4a16_gate_up(const moe_w4a16_shape* shape, const uint16_t* x,
                                                 const moe_w4a16_routing* routing, const moe_w4a16_weights* weights,
                                                 void* workspace, size_t workspace_bytes, void* stream);
MOE_W4A16_API moe_w4a16_status moe_w4a16_down(const moe_w4a16_shape* shape, const moe_w4a16_routing* routing,
                                              const moe_w4a16_weights* weights, void* workspace,
                                              size_t workspace_bytes, void* stream);
MOE_W4A16_API moe_w4a16_status moe_w4a16_combine(const moe_w4a16_shape* shape, const moe_w4a16_routing* routing,
                                                 const float* norm_gamma, float norm_eps, uint16_t* out,
                                                 void* workspace, size_t workspace_bytes, void* stream);

/* Copies the workspace's sticky error word to the host after synchronising
 * `stream`: MOE_W4A16_OK, or MOE_W4A16_ERR_TIMEOUT if a device-side wait of an
 * earlier call gave up (its outputs are then invalid).  Cleared by
 * moe_w4a16_workspace_init. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_read_error(const void* workspace, size_t workspace_bytes, void* stream,
                                      moe_w4a16_status* device_status);

/* ---- the MoE block around the layer ------------------------------------------
 * A pre-norm residual block (model card "srswti/axe-diffusion-ksl-xe", "the
 * kernels we built": the RMSNorm of a block in one launch; "what the model is":
 * a router picks each token's top-8 of 128 experts):
 *   u       = fp16(gamma * (x * r)),  r = 1 / sqrt(ss / d + eps),  ss = sum_k x_k^2
 *   logits  = u . Wr^T                 (Wr fp16 [E][d], fp32 results [T][E])
 *   out     = fp16(x + layer(u))       (layer: route + experts + combine, fp32 sum
 *                                       with x before the one rounding)
 * The logits decide the routing, so ss and the logits are defined in fp32 with
 * one fixed order of operations and are reproducible bit for bit off the GPU:
 * the d columns are dealt to 32 lanes in 8-column chunks (lane l takes chunks
 * l, l + 32, ..., in that order), each lane accumulates fmaf(a_k, b_k, acc)
 * column by column from 0, and the 32 lane sums meet in an xor butterfly
 * (offsets 16, 8, 4, 2, 1); r, x_k * r and gamma_k * (x_k * r) are single IEEE
 * fp32 operations and u rounds to nearest even.  d must be a multiple of 256
 * (ERR_SHAPE otherwise); norm_eps >= 0 and finite (ERR_VALUE).
 *
 * moe_w4a16_block_front: the pre-norm and the router projection alone.
 *   x         fp16 [T][d], read       norm_gamma  fp32 [d], read
 *   router_w  fp16 [E][d], read       u  fp16 [T][d], written    logits  fp32 [T][E], written
 * moe_w4a16_block: the whole block on `stream`: the front (u and the logits go to
 * the workspace), moe_w4a16_route on the logits (routing is written as that call
 * writes it), the experts on u and the combine with the residual.
 *   out  fp16 [T][d], written; may be x itself (each element is read before it is
 *        written by the same thread), must not overlap the workspace or routing.
 * Weights, workspace and routing follow the rules of moe_w4a16_forward. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_block_front(const moe_w4a16_shape* shape, const uint16_t* x,
                                                     const float* norm_gamma, float norm_eps,
                                                     const uint16_t* router_w, uint16_t* u, float* logits,
                                                     void* stream);
MOE_W4A16_API moe_w4a16_status moe_w4a16_block(const moe_w4a16_shape* shape, const uint16_t* x,
                                               const float* norm_gamma, float norm_eps, const uint16_t* router_w,
                                               const moe_w4a16_routing* routing, const moe_w4a16_weights* weights,
                                               uint16_t* out, void* workspace, size_t workspace_bytes,
                                               void* stream);

/* ---- per-step sampler ------------------------------------------------------
 * One denoising step's sampling over a canvas (model card
 * "srswti/axe-diffusion-ksl-xe", "the kernels we built": the entropy once per
 * step in a single streaming pass over the logits, one Gumbel-max kernel instead
 * of softmax + multinomial; "lablup/mlxcel block-diffusion docs", "Samplers":
 * the two acceptance rules).  Per position p, with t_v = logits[p][v] * inv_temperature:
 *   entropy[p]  H = -sum_v q_v ln q_v of q = softmax(t)                    (fp32)
 *   pmax[p]     max_v q_v                                                  (fp32)
 *   token[p]    a Gumbel-max draw from q, in one of two forms (cfg.noise):
 *               noise 0 (one Gumbel per group of four, the default): group g holds
 *                 entries 4g .. 4g+3; its key is fl(fl(m + ln S) + G_g) with
 *                 t_i = fl(l_i inv_temperature), m = max t_i, e_i = exp(fl(t_i - m)),
 *                 S = ((e_0 + e_1) + e_2) + e_3, G_g = -ln(-ln U_g); the winning group
 *                 is the argmax (ties to the lower g) and the token inside it the
 *                 first i with fl(..fl(e_0 + e_1).. + e_i) > fl(U'_g S) (if none, the
 *                 last i with e_i > 0).  U_g / U'_g come from word r / 256, r = g % 1024,
 *                 of Philox4x32-10 at counter (256 (g / 1024) + r % 256, p, step, 0 / 1).
 *                 The maximum of the four per-token keys below is Gumbel around
 *                 ln sum_i e^(t_i) and falls on i with probability proportional to e^(t_i)
 *                 (max-stability of the Gumbel law), so both forms sample q;
 *               noise 1 (one Gumbel per token): argmax_v (t_v + G_v), ties to the lower
 *                 v; G_v = -ln(-ln U_v), U_v from word v % 4 of Philox4x32-10 at
 *                 counter (v / 4, p, step, 0), key fma(logit, inv_temperature, G_v).
 *               U = ((x & 0x7fffff) + 1/2) 2^-23 of a word x; Philox4x32-10 (Salmon et
 *               al., SC'11) under key (seed & 0xffffffff, seed >> 32).  Every key is
 *               evaluated in fp32 with one IEEE rounding per step (the natural log as
 *               range reduction plus the atanh series to s^11, the exponential as range
 *               reduction plus the Taylor series to r^7, 0 below -87), so the token is
 *               reproducible bit for bit off the GPU
 *   accept[p]   rule 0 (entropy bound): among positions with revealed[p] == 0,
 *               sorted by (entropy, p), sorted position i is accepted iff
 *               fl(c_i - x_i) <= bound, c_i / x_i the fp32 running sum / maximum of
 *               the sorted entropies (the mlx-vlm rule (cumsum - cummax) <= bound),
 *               and the first one always;
 *               rule 1 (confidence): revealed[p] == 0 and pmax[p] > bound; if no
 *               such position, the unrevealed one with the largest pmax (ties to
 *               the lower p).  Revealed positions are never accepted.
 * Accuracy: entropy and pmax come from fp32 streaming sums; t2 = t log2 e is rounded
 * once, so with T = max |t2| of a position their relative error is about 2e-5 +
 * 2^-22 T (the tokens are exact at any scale).
 * Non-finite logits give unspecified (but in-bounds) results. */
typedef struct {
  int32_t positions;      /* P, 1 .. 1024 */
  int32_t vocab;          /* V, a multiple of 4, 4 .. 2^30 */
  float inv_temperature;  /* > 0 and finite */
  int32_t rule;           /* 0 = entropy bound, 1 = confidence threshold */
  float bound;            /* entropy bound (rule 0) or confidence threshold (rule 1), finite */
  uint32_t step;          /* denoising step: third Philox counter word */
  int32_t noise;          /* 0 = one Gumbel per group of four entries (default), 1 = one per token */
  uint64_t seed;          /* Philox key */
} moe_w4a16_sampler;

/* Device workspace bytes moe_w4a16_sample needs (0 on an invalid config). */
MOE_W4A16_API size_t moe_w4a16_sampler_workspace_bytes(const moe_w4a16_sampler* cfg);

/* Runs the sampler on `stream` (two launches).  Device pointers:
 *   logits    fp32 [P][V], 16-byte aligned        revealed  uint8 [P] (nonzero = already revealed)
 *   token     int32 [P], entropy fp32 [P], pmax fp32 [P] (4-byte aligned), accept uint8 [P]
 *   workspace moe_w4a16_sampler_workspace_bytes(cfg) bytes, 16-byte aligned (scratch, no state)
 * ERR_SHAPE on an invalid config, ERR_NULL / ERR_ALIGN / ERR_WORKSPACE as elsewhere. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_sample(const moe_w4a16_sampler* cfg, const float* logits,
                                                const uint8_t* revealed, int32_t* token, float* entropy,
                                                float* pmax, uint8_t* accept, void* workspace,
                                                size_t workspace_bytes, void* stream);

/* ---- host-side weight helpers (no GPU needed) ---------------------------- */

/* Canonical packing of uint4 codes (dg-w4a16-v1 style, model card
 * "requirements": two nibbles per byte): codes [rows][K] with values 0..15 ->
 * packed [rows][K/2], byte b of a row holding column 2b in its low nibble and
 * column 2b+1 in its high nibble.  K must be even.  ERR_VALUE if a code > 15. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_pack(const uint8_t* codes, int64_t rows, int64_t K, uint8_t* packed);

/* Inverse of moe_w4a16_pack. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_unpack(const uint8_t* packed, int64_t rows, int64_t K, uint8_t* codes);

/* Bytes of the prepared layout of one projection of all E experts:
 * exactly the canonical bytes (packed nibbles + fp16 scale + fp16 zero). */
MOE_W4A16_API size_t moe_w4a16_prepared_bytes(const moe_w4a16_shape* shape, int32_t which);

/* Rearranges one projection of all E experts from the canonical layout into the
 * kernels' prepared layout (a byte permutation; no value changes).  Host memory.
 *   which   MOE_W4A16_GATE_UP: rows R = 2f (rows [0,f) gate, [f,2f) up), K = d, g = g1
 *           MOE_W4A16_DOWN:    rows R = d, K = f, g = g2
 *   q       canonical packed codes [E][R][K/2]
 *   scale   fp16 bits [E][R][K/g]
 *   zero    fp16 bits [E][R][K/g]: the zero-point (format 0) or the bias (format 1);
 *           ignored and may be NULL for format 2 (the layout then holds 8)
 *   out     moe_w4a16_prepared_bytes(shape, which) bytes
 * ERR_VALUE if |scale| > 32 or not finite, if a zero-point is outside [0, 16]
 * (format 0) or a bias outside [-1024, 1024] (format 1).
 * The prepared layout is private to this library version: per block of 128 GEMM
 * rows, a stream of 128-column stages (the last of 64 columns when K is an odd
 * multiple of 64), each split into eight strips of 16 rows, one per compute warp;
 * a strip holds its rows' scale/zero pairs for the groups of the stage followed by
 * the codes, each 32-bit word one m16n8k16 A fragment of one lane.
 * ERR_VALUE if a scale is not finite or |scale| > 32, or a zero-point lies outside
 * [0, 16] (the kernels' fp16 dequantisation is exact only in that range). */
MOE_W4A16_API moe_w4a16_status moe_w4a16_prepare(const moe_w4a16_shape* shape, int32_t which, const uint8_t* q,
                                   const uint16_t* scale, const uint16_t* zero, uint8_t* out);

/* Inverse of moe_w4a16_prepare (for checking a prepared buffer). */
MOE_W4A16_API moe_w4a16_status moe_w4a16_unprepare(const moe_w4a16_shape* shape, int32_t which, const uint8_t* prepared,
                                     uint8_t* q, uint16_t* scale, uint16_t* zero);

/* ---- allocation-free forward ---------------------------------------------
 *
 * moe_w4a16_forward_noalloc computes exactly what moe_w4a16_forward computes
 * (the gate_up and down GEMMs and the combine, on a routing written by
 * moe_w4a16_route; the same shape rules, reduction orders and weight formats,
 * and bit-identical outputs), but keeps its scratch memory in a static device
 * array built into the library instead of a caller-provided workspace, and
 * allocates nothing.
 * The pages describe no counterpart to this call; it exists for callers that
 * cannot obtain device memory of their own -- for example a plugin running
 * inside a host application whose memory manager owns the whole device heap
 * and forbids side allocations, or a latency-critical serving loop that must
 * not call cudaMalloc because an allocation can synchronise the device and
 * stall the work already queued on it.
 *
 *   - The array holds MOE_W4A16_NOALLOC_SCRATCH_BYTES (40 MiB) and is reserved
 *     on every GPU that loads the library until the process exits.
 *   - A shape whose moe_w4a16_workspace_bytes() exceeds that size is rejected
 *     with MOE_W4A16_ERR_WORKSPACE before anything is launched (a 256-token
 *     canvas with d = 2048, f = 704 and top-8 needs about 28 MB and fits; a
 *     1024-token batch of that layer does not).
 *   - The first call on a device performs a one-time set-up on that device (it
 *     looks up the array's device address and sets kernel attributes); make
 *     that first call before capturing any stream into a CUDA graph.
 *   - Every call on a device uses the same array: calls whose GPU work may
 *     overlap (other streams, concurrently launched graphs) race with each
 *     other and give undefined results.  Each call clears the array's work
 *     counters when it starts; the rest keeps the last call's contents until
 *     overwritten.
 *   - A device-side wait that runs out records MOE_W4A16_ERR_TIMEOUT in the
 *     static array's error word (the call's output is then invalid);
 *     moe_w4a16_noalloc_read_error reads that word back.
 * Arguments are those of moe_w4a16_forward, without the workspace. */
#define MOE_W4A16_NOALLOC_SCRATCH_BYTES ((size_t)40 << 20)
MOE_W4A16_API moe_w4a16_status moe_w4a16_forward_noalloc(const moe_w4a16_shape* shape, const uint16_t* x,
                                                         const moe_w4a16_routing* routing,
                                                         const moe_w4a16_weights* weights, const float* norm_gamma,
                                                         float norm_eps, uint16_t* out, void* stream);

/* Copies the error word of the current device's static array to
 * *device_status after synchronising `stream`: MOE_W4A16_OK, or the status of a
 * device-side failure of the last moe_w4a16_forward_noalloc call on this device
 * (each such call clears the word when it starts).  Errors: ERR_NULL for a NULL
 * device_status, ERR_DEVICE on a device other than compute capability 10.3,
 * ERR_CUDA if the copy fails. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_noalloc_read_error(void* stream, moe_w4a16_status* device_status);

/* Self-test of the device-side failure path.  Every wait in the expert launch
 * (on its mbarrier rings and on the counters other CTAs raise) is bounded: on
 * expiry the kernel records MOE_W4A16_ERR_TIMEOUT in the workspace's error
 * word, every role of the CTA leaves its loop, in-flight copies are drained and
 * the kernel returns, so the context stays usable.  This call launches one warp
 * that runs the same wait helpers, with bound limit_ns, on an mbarrier phase
 * that nothing completes and on a workspace counter that nothing raises; both
 * give up and moe_w4a16_read_error then reports MOE_W4A16_ERR_TIMEOUT (clear it
 * with moe_w4a16_workspace_init).  The workspace must have been initialised.
 *   limit_ns  1 .. 2e9 (ERR_VALUE otherwise); the call takes about 2 limit_ns on the device. */
MOE_W4A16_API moe_w4a16_status moe_w4a16_selftest_wait_timeout(void* workspace, size_t workspace_bytes,
                                                               uint64_t limit_ns, void* stream);

/* Static description of a status code (never NULL). */
MOE_W4A16_API const char* moe_w4a16_status_string(moe_w4a16_status status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_W4A16_H */
