/*
 * ito.h -- C ABI of the integer-only training library for one GB300 GPU
 * (sm_103a).
 *
 * What it computes: the NITI integer training step -- int8 x int8 -> int32
 * contractions for the forward pass, delta propagation and weight gradient,
 * each followed by a per-tensor dynamic-shift requantisation, and the NITI
 * integer weight update -- as described in "Integer On-Device Training:
 * Overview" (TI C2000 MCU AI user guide), section 3 "The NITI Algorithm",
 * "The Solution: Dynamic Shifts", Steps 1-5:
 *
 *   max_val  = max |G|                                   (Step 1)
 *   shift    = max(0, ceil(log2(max_val + 1)) - target_bits)   (Step 2)
 *   Gq       = round-half-up(G >> shift), saturated to int8     (Step 3)
 *   wshift   = max(0, shift - mu_weight)                 (Step 4)
 *   W        = sat_int8(W - round-half-up(Gq >> wshift)) (Steps 4-5)
 *
 * Conventions (all entry points):
 *  - Tensors are row-major. Linear weights are indexed W[oc * IC + ic]
 *    (TiGrIS "Compilation Pipeline", pass 3 "Matrix product relabel");
 *    activations are [B][features]; conv activations are NHWC and conv weights
 *    [OC][3][3][IC] (the same page, emission stage "Layout transpose").
 *  - Tensor pointers are DEVICE pointers owned by the caller unless an entry
 *    point says "host". The library never frees them and never keeps them after
 *    the call returns (a model keeps only memory it allocated itself).
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream). Calls only enqueue work on it and return before it runs, unless
 *    the entry point says it synchronises.
 *  - Max and shift scalars stay on the device, in caller buffers.
 *  - Return value: an ito_status. ITO_ERR_ARG / ITO_ERR_SHAPE are detected on
 *    the host before anything is enqueued; ITO_ERR_CUDA reports a failed launch
 *    or runtime call (ito_last_error_string() gives its text). Kernels never
 *    trap: a failure they detect (a bounded wait that gave up) is written to a
 *    per-device error word that ito_get_error() reads and clears.
 *  - Rounding "round-half-up" is floor(x / 2^s + 1/2): ties go toward +inf.
 *    sat_int8 clamps to [-128, 127].
 */
#ifndef ITO_H
#define ITO_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ito_status {
    ITO_OK = 0,
    ITO_ERR_ARG = 1,          /* null or misaligned pointer, unknown enum value */
    ITO_ERR_SHAPE = 2,        /* non-positive, inconsistent or too large size */
    ITO_ERR_CUDA = 3,         /* a CUDA launch or runtime call failed */
    ITO_ERR_TIMEOUT = 4,      /* a kernel's bounded wait gave up (device error word) */
    ITO_ERR_EXPONENT = 5,     /* a DFP16 shared exponent left the signed 8-bit range */
    ITO_ERR_UNSUPPORTED = 6   /* a valid request this library does not implement */
} ito_status;

/* NITI parameters: target_bits (7 for int8 tensors) and mu_weight (the
 * learning-rate control of Step 4). */
typedef struct ito_niti_params {
    int32_t target_bits;
    int32_t mu_weight;
} ito_niti_params;

/* ------------------------------------------------------------------------
 * Library state
 * ---------------------------------------------------------------------- */

/* Reads and clears the current device's error word (ITO_OK if no kernel
 * reported a failure). Synchronises the device. */
int ito_get_error(void);

/* Text of the last ITO_ERR_CUDA / ITO_ERR_ARG / ITO_ERR_SHAPE raised on this
 * host thread; never NULL. */
const char *ito_last_error_string(void);

/* Library version, for the Python binding's sanity check. */
int ito_version(void);

/* Self-test of failure detection (the pages have no counterpart): launches one
 * CTA that waits on an mbarrier nothing completes, with the bounded wait every
 * pipeline barrier of the contraction kernels uses. After the wait's limit
 * (2 s) the kernel records ITO_ERR_TIMEOUT in the device error word and
 * returns; the call synchronises `stream` and returns ITO_OK, and
 * ito_get_error() then reports ITO_ERR_TIMEOUT. No GPU fault, trap or hang is
 * involved; the context stays usable. Errors: ITO_ERR_CUDA. */
int ito_selftest_wait_timeout(void *stream);

/* ------------------------------------------------------------------------
 * Single-layer operations (int8 Linear layer, NITI)
 *
 * Contractions run on the tensor cores with bf16 operands that hold the int8
 * values exactly; sums are exact (fp32 accumulation over K chunks of at most
 * 1024 terms, each chunk's integer result added in int32). A caller workspace
 * of ito_linear_workspace_size() bytes holds the bf16 operand copies.
 * ---------------------------------------------------------------------- */

/* Bytes of device workspace any of ito_linear_fwd / _bwd_delta / _wgrad needs
 * for these sizes (0 on invalid sizes): the bf16 operand copies, plus room for
 * int32 partial results when a contraction with few output tiles and a long
 * K is split along K across SMs (partials summed exactly afterwards). */
size_t ito_linear_workspace_size(int B, int IC, int OC);

/* Forward contraction + requantisation of one Linear layer ("Integer
 * On-Device Training: Overview", section 3, Steps 1-3 applied to the layer
 * output; section 7 layer types Linear and Linear+ReLU):
 *   y32[b][oc] = sum_ic x[b][ic] * W[oc][ic]        (int32, exact)
 *   *d_max     = max |y32|   (uint32; |INT32_MIN| = 2^31 fits)
 *   *d_shift   = max(0, bitlen(*d_max) - p.target_bits)
 *   y[b][oc]   = sat_int8(round-half-up(y32 >> shift)), then max(0, .) if relu
 * x: int8 [B][IC]; W: int8 [OC][IC]; y32: int32 [B][OC]; y: int8 [B][OC].
 * d_max, d_shift: one device scalar each. workspace: device, 256-byte
 * aligned, workspace_bytes >= ito_linear_workspace_size(B, IC, OC).
 * Errors: ITO_ERR_ARG (null pointer, misaligned workspace),
 * ITO_ERR_SHAPE (B, IC or OC < 1, or a contraction length above 2^20). */
int ito_linear_fwd(const int8_t *x, const int8_t *W, int B, int IC, int OC, int relu,
                   ito_niti_params p, void *workspace, size_t workspace_bytes,
                   int32_t *y32, uint32_t *d_max, int32_t *d_shift, int8_t *y, void *stream);

/* Bytes of the scratch array built into the library for
 * ito_linear_fwd_noalloc (16 MiB). */
#define ITO_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/* ito_linear_fwd without a workspace argument, for callers that cannot
 * allocate device memory while they run -- for example code inside a CUDA
 * host callback (where CUDA calls that allocate are not permitted), or a
 * plug-in whose host framework owns all device memory and forbids allocation
 * in its execute hook. The pages have no counterpart to this entry point.
 *
 * It computes exactly what ito_linear_fwd computes, with the same arguments
 * minus workspace/workspace_bytes, and allocates nothing: its scratch (the
 * bf16 copies of x and W, rows padded to 8 elements, each copy rounded up to
 * 256 bytes) is a fixed device array of ITO_NOALLOC_SCRATCH_BYTES inside the
 * library, which every GPU that loads the library holds until the process
 * exits. (It never splits the contraction along K.)
 *  - Sizes whose scratch need exceeds ITO_NOALLOC_SCRATCH_BYTES are rejected
 *    with ITO_ERR_SHAPE before anything is enqueued.
 *  - The first call on a device looks up the array's device address on that
 *    device (the device must be current); make that first call before any
 *    stream capture. The address is kept per device context: after a
 *    cudaDeviceReset the next call on that device looks it up again, so make
 *    that call, too, before any stream capture.
 *  - All calls share the array: calls whose work overlaps on the GPU (for
 *    instance on two streams without ordering) race on it. Serialise them.
 * Outputs, errors and stream semantics as ito_linear_fwd. */
int ito_linear_fwd_noalloc(const int8_t *x, const int8_t *W, int B, int IC, int OC, int relu,
                           ito_niti_params p, int32_t *y32, uint32_t *d_max, int32_t *d_shift,
                           int8_t *y, void *stream);

/* Delta propagation of one Linear layer (same page, the note under Step 5:
 * the propagated delta is requantised to target_bits = 7 so it fits int8),
 * gated by the ReLU of the layer below:
 *   d32[b][ic]      = sum_oc delta[b][oc] * W[oc][ic]    (int32, exact)
 *   *d_max, *d_shift as in ito_linear_fwd
 *   delta_prev[b][ic] = (a_prev == NULL || a_prev[b][ic] > 0)
 *                        ? sat_int8(round-half-up(d32 >> shift)) : 0
 * delta: int8 [B][OC]; W: int8 [OC][IC] (the weights before this step's
 * update); a_prev: int8 [B][IC] or NULL; d32: int32 [B][IC];
 * delta_prev: int8 [B][IC]. Errors as ito_linear_fwd. */
int ito_linear_bwd_delta(const int8_t *delta, const int8_t *W, const int8_t *a_prev, int B, int IC,
                         int OC, ito_niti_params p, void *workspace, size_t workspace_bytes,
                         int32_t *d32, uint32_t *d_max, int32_t *d_shift, int8_t *delta_prev,
                         void *stream);

/* Weight gradient of one Linear layer, summed over the batch (the
 * "accumulated gradient tensor G for one weight matrix" of Step 1):
 *   G[oc][ic] = sum_b delta[b][oc] * a_prev[b][ic]    (int32, exact)
 *   *d_max    = max |G|
 * delta: int8 [B][OC]; a_prev: int8 [B][IC] (the layer's input);
 * G: int32 [OC][IC]. Errors as ito_linear_fwd. */
int ito_linear_wgrad(const int8_t *delta, const int8_t *a_prev, int B, int IC, int OC,
                     void *workspace, size_t workspace_bytes, int32_t *G, uint32_t *d_max,
                     void *stream);

/* NITI weight update, Steps 2-5, in place (reading of Step 4: its operand is
 * G_quantized, the tensor already shifted and saturated in Step 3):
 *   s = max(0, bitlen(*d_max) - p.target_bits); ws = max(0, s - p.mu_weight)
 *   W[i] = sat_int8(W[i] - round-half-up(sat_int8(round-half-up(G[i] >> s)) >> ws))
 * W: int8 [n] (updated in place); G: int32 [n]; d_max: max|G| (as written
 * by ito_linear_wgrad). d_shift, d_wshift: device scalars receiving s and
 * ws (may be NULL). d_nonzero: device uint32 to which the number of nonzero
 * weight steps is ADDED (may be NULL; the caller zeroes it).
 * Errors: ITO_ERR_ARG (null W, G or d_max), ITO_ERR_SHAPE (n < 1). */
int ito_niti_update(int8_t *W, const int32_t *G, int64_t n, const uint32_t *d_max,
                    ito_niti_params p, int32_t *d_shift, int32_t *d_wshift, uint32_t *d_nonzero,
                    void *stream);

/* Top error written by the user's compute_loss ("Integer On-Device Training:
 * Overview", section 4: compute_loss reads the int8 logits and writes dy):
 *   delta[b][j] = sat_int8(logits[b][j] - target_mag * [j == labels[b]])
 * logits: int8 [B][C]; labels: int32 [B] in [0, C); delta: int8 [B][C].
 * A label outside [0, C) has no class to take the target: the kernel copies
 * that row and records ITO_ERR_ARG in the device error word (ito_get_error).
 * Errors: ITO_ERR_ARG, ITO_ERR_SHAPE. */
int ito_top_error(const int8_t *logits, const int32_t *labels, int B, int C, int32_t target_mag,
                  int8_t *delta, void *stream);

/* ------------------------------------------------------------------------
 * Single-layer operations: 3x3 Conv2D (+ReLU) and global integer pooling
 * ("Integer On-Device Training: Overview", section 7: Conv2D and Conv2D+ReLU
 * layers, dense, groups = 1, dilation = 1). Activations are NHWC, conv
 * weights [OC][3][3][IC] (the channel-last layout of the TiGrIS "Compilation
 * Pipeline" page, emission stage); padding is 1, so OH = (H - 1) / stride + 1
 * and OW = (W - 1) / stride + 1. A conv is the Linear contraction over the
 * im2col patch matrix [B*OH*OW][9*IC] in (kh, kw, ic) order; sums are exact
 * as for the Linear operations.
 * ---------------------------------------------------------------------- */

/* Bytes of device workspace any of ito_conv2d_fwd / _bwd_delta / _wgrad
 * needs for these sizes (0 on invalid sizes): bf16 patch, weight and delta
 * copies, the int32 patch-space delta, split-K partials and one scratch word.
 * A stride-2 conv with even H and W, OW = W/2 of 8, 16 or 32, OH = H/2 a power
 * of two with OH*OW >= 32, and IC, OC multiples of 64 is contracted without
 * patches (the input's bf16 copy is read through its four parity planes, the
 * propagated delta by its four parity phases); it uses the same workspace
 * (the patch slot holds the input's bf16 copy) and gives the same results. */
size_t ito_conv2d_workspace_size(int B, int H, int W, int IC, int OC, int stride);

/* Forward 3x3 conv + requantisation:
 *   y32[b][oh][ow][oc] = sum_{kh,kw,ic} x[b][oh*stride-1+kh][ow*stride-1+kw][ic] * Wt[oc][kh][kw][ic]
 *                        (taps outside the input are 0)
 *   *d_max, *d_shift, y as in ito_linear_fwd (ReLU when relu != 0).
 * x: int8 [B][H][W][IC]; Wt: int8 [OC][3][3][IC]; y32: int32 [B][OH][OW][OC];
 * y: int8 [B][OH][OW][OC]. workspace: device, 256-byte aligned, at least
 * ito_conv2d_workspace_size() bytes.
 * Errors: ITO_ERR_ARG (null pointer, workspace misaligned or too small),
 * ITO_ERR_SHAPE (a size < 1, stride outside 1..4, IC above 2^16, OC above
 * 2^20, or B*OH*OW above 2^20). */
int ito_conv2d_fwd(const int8_t *x, const int8_t *Wt, int B, int H, int W, int IC, int OC, int stride,
                   int relu, ito_niti_params p, void *workspace, size_t workspace_bytes, int32_t *y32,
                   uint32_t *d_max, int32_t *d_shift, int8_t *y, void *stream);

/* Delta propagation of a 3x3 conv, gated by the ReLU of the layer below:
 *   d32[b][ih][iw][ic] = sum over (oh, ow, kh, kw) with oh*stride-1+kh = ih and
 *                        ow*stride-1+kw = iw of delta[b][oh][ow][oc] * Wt[oc][kh][kw][ic]
 *                        (the transpose of the forward; int32, exact)
 *   *d_max = max |d32|; *d_shift and delta_prev as in ito_linear_bwd_delta.
 * delta: int8 [B][OH][OW][OC]; Wt: the weights before this step's update;
 * a_prev: int8 [B][H][W][IC] or NULL; d32: int32 [B][H][W][IC];
 * delta_prev: int8 [B][H][W][IC]. Errors as ito_conv2d_fwd. */
int ito_conv2d_bwd_delta(const int8_t *delta, const int8_t *Wt, const int8_t *a_prev, int B, int H,
                         int W, int IC, int OC, int stride, ito_niti_params p, void *workspace,
                         size_t workspace_bytes, int32_t *d32, uint32_t *d_max, int32_t *d_shift,
                         int8_t *delta_prev, void *stream);

/* Weight gradient of a 3x3 conv, summed over the batch and the output
 * positions:
 *   G[oc][kh][kw][ic] = sum_{b,oh,ow} delta[b][oh][ow][oc] * x[b][oh*stride-1+kh][ow*stride-1+kw][ic]
 *   *d_max = max |G|
 * delta: int8 [B][OH][OW][OC]; x: int8 [B][H][W][IC] (the layer input);
 * G: int32 [OC][3][3][IC]. Errors as ito_conv2d_fwd. */
int ito_conv2d_wgrad(const int8_t *delta, const int8_t *x, int B, int H, int W, int IC, int OC,
                     int stride, void *workspace, size_t workspace_bytes, int32_t *G, uint32_t *d_max,
                     void *stream);

/* Global integer sum pooling + requantisation without ReLU (no division: the
 * NITI shift that follows rescales the sum):
 *   P32[b][c] = sum_pos a[b][pos][c];  *d_max = max |P32|;
 *   *d_shift = max(0, bitlen(*d_max) - p.target_bits);
 *   pa[b][c] = sat_int8(round-half-up(P32 >> shift))
 * a: int8 [B][HW][C] (NHWC with HW = H*W); P32: int32 [B][C]; pa: int8 [B][C].
 * Errors: ITO_ERR_ARG (null pointer), ITO_ERR_SHAPE (a size < 1, HW above 2^24). */
int ito_gap_fwd(const int8_t *a, int B, int HW, int C, ito_niti_params p, int32_t *P32,
                uint32_t *d_max, int32_t *d_shift, int8_t *pa, void *stream);

/* Backward of the pooling: the pooled delta is broadcast to every position,
 * gated by the ReLU of the pooled layer (no rescale):
 *   delta[b][pos][c] = (a[b][pos][c] > 0) ? dP[b][c] : 0
 * dP: int8 [B][C]; a: int8 [B][HW][C]; delta: int8 [B][HW][C].
 * Errors: ITO_ERR_ARG, ITO_ERR_SHAPE (a size < 1). */
int ito_gap_bwd(const int8_t *dP, const int8_t *a, int B, int HW, int C, int8_t *delta, void *stream);

/* ------------------------------------------------------------------------
 * Models: a sequential stack of trainable layers ("Integer On-Device
 * Training: Overview", section 4: INT_LAYERS[], an array of layer descriptors
 * with mutable int8 weights; INTODT_Forward / INTODT_Backward / INTODT_Infer).
 * A model owns all its device memory (allocated at creation, nothing is
 * allocated per step) and keeps every intermediate tensor of the last step.
 * ---------------------------------------------------------------------- */

typedef enum ito_layer_kind {
    ITO_LAYER_LINEAR = 0,        /* Linear producing logits (last layer) */
    ITO_LAYER_LINEAR_RELU = 1,   /* Linear + ReLU */
    ITO_LAYER_CONV3X3_RELU = 2,  /* 3x3 Conv2D + ReLU, pad 1, NHWC, weights [OC][3][3][IC] */
    ITO_LAYER_GAP = 3            /* global integer sum pooling + requantisation (no weights) */
} ito_layer_kind;

typedef struct ito_layer_desc {
    int32_t kind;          /* ito_layer_kind */
    int32_t in_features;   /* IC (channels for conv / GAP) */
    int32_t out_features;  /* OC (ignored for GAP: equals in_features) */
    int32_t in_h, in_w;    /* spatial input size (conv / GAP); 0 for Linear */
    int32_t stride;        /* conv stride (1 or 2); 0 otherwise */
} ito_layer_desc;

typedef struct ito_model ito_model;

/* Creates a model on the current device. The stack must be a sequence of
 * conv layers, optionally one GAP, then Linear(+ReLU) layers ending with one
 * ITO_LAYER_LINEAR. Weights start at zero (set them with
 * ito_model_set_weights). target_mag: the integer target of the true class
 * in the top error (64).
 * Errors: ITO_ERR_ARG, ITO_ERR_SHAPE (inconsistent sizes),
 * ITO_ERR_UNSUPPORTED (a layer order outside the one above), ITO_ERR_CUDA
 * (allocation failed). */
int ito_model_create(const ito_layer_desc *layers, int n_layers, int batch, ito_niti_params p,
                     int32_t target_mag, ito_model **out);

/* Options of ito_model_create_ex ("Integer On-Device Training: Overview",
 * section 5 "Full Model vs Partial Model" and section 8 "Memory
 * Considerations"):
 *  - input_uint8: the first layer (a Linear) receives UINT8 activations in
 *    [0, 255], as from a frozen prefix whose last layer has a ReLU;
 *  - trainable_from: layers before this index are frozen (forward only: no
 *    weight gradient, no update, and no delta is propagated into them) --
 *    trainable_layers_from_last = n_layers - trainable_from;
 *  - packed_masks: the ReLU masks of the backward pass are kept bit-packed,
 *    ceil(out_size / 8) bytes per sample and ReLU layer (each such layer's
 *    output width must be a multiple of 8);
 *  - pingpong_grads: the deltas of all layers share two buffers ("Grad
 *    Buffers": two ping-pong buffers sized batch * the largest layer output)
 *    instead of one per layer; layer l's delta lives in buffer l % 2, so after
 *    a step only the deltas of layers 0 and 1 remain readable (the tensor
 *    names e<l> of higher layers alias them);
 *  - speculate_min_elems: speculative requantisation (ito_model_set_speculation)
 *    covers only the contractions whose output has at least this many
 *    elements; 0 = 4,194,304. Below that the requantisation pass is a few
 *    microseconds and the re-launch, with its occasional recomputation, costs
 *    more than it saves. */
typedef struct ito_model_options {
    int32_t input_uint8;
    int32_t trainable_from;
    int32_t packed_masks;
    int32_t pingpong_grads;
    int32_t speculate_min_elems;
} ito_model_options;

/* ito_model_create with options (NULL = all zero, the same as
 * ito_model_create). Errors: as ito_model_create; ITO_ERR_UNSUPPORTED for a
 * UINT8 input to a conv layer or packed masks on a width not a multiple of 8;
 * ITO_ERR_ARG for trainable_from outside [0, number of weight layers). */
int ito_model_create_ex(const ito_layer_desc *layers, int n_layers, int batch, ito_niti_params p,
                        int32_t target_mag, const ito_model_options *opt, ito_model **out);

/* Frees the model's device memory. Synchronises the device. NULL is a no-op. */
int ito_model_destroy(ito_model *m);

/* Copies weights of trainable layer `layer` (counted over layers that have
 * weights) in or out. W points to int8 [OC][IC] or [OC][3][3][IC]; host
 * memory if `on_host` != 0, else device memory. Enqueued on `stream`; with
 * host memory the call synchronises the stream. */
int ito_model_set_weights(ito_model *m, int layer, const int8_t *W, int on_host, void *stream);
int ito_model_get_weights(const ito_model *m, int layer, int8_t *W, int on_host, void *stream);

/* Looks up a named device tensor of the last step (names as in the CPU
 * oracle: "y0" int32 forward contraction of layer 0, "a0" its int8 output,
 * "m0" its bit-packed ReLU mask (packed_masks models),
 * "e0" int8 delta at the output of layer 0, "d1" int32 delta-propagation
 * contraction of layer 1, "g0" int32 weight gradient, "w0" int8 weights,
 * "stats" int32 scalars; see ito_model_stat_index; "spec" int32 [8 * layers]:
 * the forward and delta-propagation shift predictions the step used, the
 * shifts the step computed, 1 where the contraction's epilogue speculates, and
 * the re-launch words (0: the prediction held, else the step's shift + 1: the
 * re-launch recomputed the outputs; 0 where the slot does not speculate), each
 * block of 2 * layers indexed by weight layer, -1 in the first two where none;
 * "spec_count"
 * int64 [2]: predictions that held and that missed since creation, scored at
 * the start of the following step (see ito_model_set_speculation)). Writes the device
 * pointer, the element type (1 = int8, 2 = int16, 4 = int32, 8 = int64) and
 * element count. The pointer stays valid until ito_model_destroy.
 * Errors: ITO_ERR_ARG (unknown name). */
int ito_model_tensor(const ito_model *m, const char *name, void **dev_ptr, int *elem_bytes,
                     int64_t *numel);

/* Static per-channel requantisation of a Linear layer's forward output, the
 * TI library's own forward ("Integer On-Device Training: Overview", section
 * 4: each layer holds INT32 offsets, mutable and updated by the backward
 * pass, and const k (shift) and mult arrays from the exported OSS chain
 * Add(offset) -> Mul -> Mul -> Floor -> Clip). Readings: the layer output is
 *   a[b][c] = clip(floor((y32[b][c] + offset[c]) * mult[c] / 2^shift[c]),
 *                  relu ? 0 : -128, 127)      (int64 product)
 * in place of the dynamic NITI shift; each step the offsets' gradient
 * g[c] = sum_b delta[b][c] updates them with NITI Steps 1-5 (saturating to
 * int32). offset, mult, shift: int32 [OC], host or device memory (on_host);
 * shift in 0..62. Names of the offsets and their gradient in
 * ito_model_tensor: "off<l>", "og<l>"; stats "ogmax<l>", "ogs<l>", "ows<l>",
 * "onz<l>". Errors: ITO_ERR_ARG, ITO_ERR_UNSUPPORTED (a conv layer). */
int ito_model_set_static_requant(ito_model *m, int layer, const int32_t *offset, const int32_t *mult,
                                 const int32_t *shift, int on_host, void *stream);

/* Position of a named scalar in the model's "stats" array (int32), e.g.
 * "ymax0", "ys0", "dmax1", "ds1", "gmax0", "gs0", "ws0", "nz0", "pmax",
 * "ps"; -1 if unknown. Max values are stored as their uint32 bit pattern. */
int ito_model_stat_index(const ito_model *m, const char *name);

/* Number of int32 entries in the stats array. */
int ito_model_num_stats(const ito_model *m);

/* One training step on one batch (device pointers): forward through all
 * layers, top error against `labels`, then for each layer from the top down:
 * delta propagation with the pre-update weights (not for the first layer),
 * weight gradient, NITI update. x: int8 [batch][in_features] (NHWC for a conv
 * first layer); labels: int32 [batch] in [0, classes) (an out-of-range label
 * records ITO_ERR_ARG in the device error word, as in ito_top_error).
 * Enqueued on `stream`; no host synchronisation. */
int ito_train_step(ito_model *m, const int8_t *x, const int32_t *labels, void *stream);

/* Replays whole training steps as CUDA graphs (enable != 0) or launches
 * every kernel directly (0, the default). With graphs on, a step called on a
 * non-default stream runs directly the first time, is captured into a graph the
 * next time for its (x, labels) pointer pair (up to 8 pairs are kept), and is
 * replayed from then on; the legacy default stream (NULL) and steps run with
 * ito_model_profile enabled always launch directly. Synchronises the device;
 * frees all captured graphs. */
int ito_model_use_graphs(ito_model *m, int enable);

/* Stream layout of the backward pass (the results are the same in every mode):
 *   0: every launch on the caller's stream;
 *   1: the requantisation of each propagated delta and the weight and offset
 *      updates run on a second, model-owned stream beside the next contractions
 *      (a bandwidth-bound pass shares the SMs with a tensor-core one);
 *   2: only the weight updates run on the second stream;
 *   3: the delta chain (delta propagation, its requantisation, the next layer's delta
 *      propagation) stays on the caller's stream and each layer's weight gradient and
 *      update run on the second stream (the weight gradients with their own split-K
 *      workspace); not with ping-pong delta buffers or static requantisation.
 * Events order every read after its write; the step ends joined on the caller's
 * stream. Changing the mode synchronises the device and drops captured graphs.
 * A new model takes mode 1, or, when every delta propagation requantises
 * speculatively (see ito_model_set_speculation), mode 3 (mode 0 where mode 3 is not
 * possible). Errors: ITO_ERR_ARG (NULL model, mode outside 0..3), ITO_ERR_UNSUPPORTED
 * (mode 3 with ping-pong delta buffers or static requantisation). */
int ito_model_set_overlap(ito_model *m, int mode);

/* Writes the model's current backward stream layout (0, 1 or 2) to *mode (a
 * scheduling control; the pages have no counterpart). Errors: ITO_ERR_ARG (NULL
 * argument). */
int ito_model_get_overlap(const ito_model *m, int *mode);

/* Speculative requantisation (on by default in a new model). NITI's shift of a tensor
 * depends on the whole tensor's max, so requantisation is a second pass over
 * the int32 result. With speculation on, the epilogue of the forward and
 * delta-propagation contractions (CTA-pair kernel; int8 row length a multiple
 * of 16; no packed masks, static requantisation or ping-pong buffers) writes
 * the requantised int8 tensor and its bf16 copy using the shift the same
 * tensor had in the previous step, and folds the max, but writes no int32
 * result. A second launch of the same contraction computes this step's shift
 * from the max in its prologue and returns at once when the prediction held;
 * otherwise (or when there was no prediction yet, as in the first step) it
 * recomputes the contraction and writes the outputs with the step's shift. The
 * int8, bf16 and scalar results are NITI's in either case; the int32 tensors
 * "y<l>" and "d<l>" of those contractions are not written while speculation is
 * on. Changing the setting synchronises the device and drops captured graphs.
 * Errors: ITO_ERR_ARG. */
int ito_model_set_speculation(ito_model *m, int enable);

/* Writes 1 to *enabled when speculative requantisation is on for this model,
 * else 0 (a scheduling control; the pages have no counterpart). Errors:
 * ITO_ERR_ARG (NULL argument). */
int ito_model_get_speculation(const ito_model *m, int *enabled);

/* The same step from HOST buffers: copies x and labels into the model's
 * device buffers, runs the step, copies the stats array (ito_model_num_stats
 * int32) back to stats_host (may be NULL), and synchronises the stream.
 * Host buffers should be pinned for full copy speed. */
int ito_train_step_host(ito_model *m, const int8_t *x_host, const int32_t *labels_host,
                        int32_t *stats_host, void *stream);

/* The training step of "Integer On-Device Training: Overview", section 4 (forward,
 * compute_loss, backward with the NITI update), from host buffers without waiting, for a
 * pipeline of steps: the copy of x_host and
 * labels_host goes on a model-owned copy stream into one of two model-owned device input
 * buffers (alternating from call to call, after the step that last read that buffer),
 * the step runs on `stream` after the copy, and the stats array (ito_model_num_stats
 * int32) is copied to stats_host (may be NULL) on `stream`. So the copy of the next
 * call's batch overlaps this step. The host buffers must be pinned for the copies to
 * be asynchronous and must not change until the copy is done (synchronising `stream`
 * after the next call, or after this one, is enough); stats_host holds this step's
 * statistics once `stream` has passed it. Errors: ITO_ERR_ARG, ITO_ERR_CUDA. */
int ito_train_step_host_async(ito_model *m, const int8_t *x_host, const int32_t *labels_host,
                              int32_t *stats_host, void *stream);

/* Forward pass only ("INTODT_Infer"): writes the int8 logits [batch][C]. */
int ito_infer(ito_model *m, const int8_t *x, int8_t *logits, void *stream);

/* Checkpoint ("Trained Weights in RAM": snapshot the weight and offset arrays
 * and restore them before training resumes): raw little-endian int8 weights
 * of every layer after a small header with the layer shapes, then per layer a
 * static-requantisation flag followed (when set) by its offsets, mult and
 * shift arrays.
 * Synchronise the device. Errors: ITO_ERR_ARG (path), ITO_ERR_SHAPE (file
 * does not match the model). */
int ito_model_save(const ito_model *m, const char *path);
int ito_model_load(ito_model *m, const char *path);

/* ------------------------------------------------------------------------
 * DFP16: dynamic fixed point tensors ("Mixed Precision Training of
 * Convolutional Neural Networks using Integer Operations", section 3 "The
 * Dynamic Fixed Point Format" and 3.1 "DFP Tensor Primitives"): an int16
 * mantissa tensor i with one shared signed 8-bit exponent E (value i * 2^E).
 * A product tensor carries exponent Ea + Eb; down-conversion to DFP16 shifts
 * right by Rs and adds Rs to the exponent.
 *
 * Readings used here (the page leaves them open): contractions are exact in
 * int64 (no 32-bit wrap); Rs = max(0, bitlen(max|P|) - 15); the shift rounds
 * half up and the mantissa saturates to [-32767, 32767]. Exponents are int32
 * device scalars holding int8 values; a result exponent outside [-128, 127]
 * raises ITO_ERR_EXPONENT in the device error word (ito_get_error).
 *
 * Contractions run on the tensor cores: each int16 is split into two bf16
 * limbs (v = 256*h + l, l in [-128, 127]), four limb products per term are
 * accumulated exactly in fp32 over chunks of 512 terms and combined in int64.
 * Workspace: ito_dfp16_workspace_size() bytes, 256-byte aligned, for the limb
 * planes of both operands.
 * ---------------------------------------------------------------------- */

size_t ito_dfp16_workspace_size(int B, int IC, int OC);

/* p64[b][oc] = sum_ic x[b][ic] * W[oc][ic] (int64, exact); *d_max = max|p64|
 * (uint64); *d_rs = Rs; y = sat16(round-half-up(p64 >> Rs)) (int16 [B][OC]);
 * *d_exp_y = *d_exp_x + *d_exp_w + Rs. x: int16 [B][IC]; W: int16 [OC][IC].
 * Errors: ITO_ERR_ARG, ITO_ERR_SHAPE. */
int ito_dfp16_linear_fwd(const int16_t *x, const int32_t *d_exp_x, const int16_t *W,
                         const int32_t *d_exp_w, int B, int IC, int OC, void *workspace,
                         size_t workspace_bytes, int64_t *p64, uint64_t *d_max, int16_t *y,
                         int32_t *d_exp_y, int32_t *d_rs, void *stream);

/* p64[b][ic] = sum_oc delta[b][oc] * W[oc][ic]; down-converted into
 * delta_prev (int16 [B][IC]) with exponent *d_exp_delta + *d_exp_w + Rs. */
int ito_dfp16_linear_bwd_delta(const int16_t *delta, const int32_t *d_exp_delta, const int16_t *W,
                               const int32_t *d_exp_w, int B, int IC, int OC, void *workspace,
                               size_t workspace_bytes, int64_t *p64, uint64_t *d_max,
                               int16_t *delta_prev, int32_t *d_exp_prev, int32_t *d_rs, void *stream);

/* p64[oc][ic] = sum_b delta[b][oc] * x[b][ic]; down-converted into g (int16
 * [OC][IC]) with exponent *d_exp_delta + *d_exp_x + Rs. */
int ito_dfp16_linear_wgrad(const int16_t *delta, const int32_t *d_exp_delta, const int16_t *x,
                           const int32_t *d_exp_x, int B, int IC, int OC, void *workspace,
                           size_t workspace_bytes, int64_t *p64, uint64_t *d_max, int16_t *g,
                           int32_t *d_exp_g, int32_t *d_rs, void *stream);

/* Integer SGD on DFP16 weights with a fixed exponent exp_w and learning rate
 * 2^-eta (a reading: the page trains with FP32 SGD): k = exp_w + eta - *d_exp_g,
 * dW = round-half-up(g >> k) for k >= 0, g * 2^-k for k < 0, then
 * W = sat16(W - dW) in place. *d_k receives k (may be NULL); the number of
 * nonzero dW is ADDED to *d_nonzero (may be NULL). W, g: int16 [n]. */
int ito_dfp16_update(int16_t *W, const int16_t *g, const int32_t *d_exp_g, int64_t n, int32_t exp_w,
                     int32_t eta, int32_t *d_k, uint32_t *d_nonzero, void *stream);

/* Float -> DFP16 ("Mixed Precision Training...", section 3.1: a floating-
 * point tensor's shared exponent is derived from its absolute maximum's
 * exponent). Reading: with max|f| = frac * 2^e (frac in [0.5, 1)), E = e - 15;
 * mant[i] = f[i] * 2^-E rounded to nearest (ties to even), saturated to
 * [-32767, 32767]; an all-zero tensor gets E = 0. f: float [n] (finite);
 * d_max_bits: device uint32 scratch (receives the bits of max|f|); mant:
 * int16 [n]; *d_exp = E. A non-finite input raises ITO_ERR_ARG and an E
 * outside int8 ITO_ERR_EXPONENT in the device error word. */
int ito_dfp16_from_float(const float *f, int64_t n, uint32_t *d_max_bits, int16_t *mant, int32_t *d_exp,
                         void *stream);

/* DFP16 -> float: f[i] = mant[i] * 2^(*d_exp), rounded once to float. */
int ito_dfp16_to_float(const int16_t *mant, const int32_t *d_exp, int64_t n, float *f, void *stream);

/* DFP16 Linear forward with an FP32 output (the page's section 4: the
 * kernels consume DFP-16 tensors and produce FP32 outputs, quantised for the
 * next layer, e.g. with ito_dfp16_from_float): p64 as in ito_dfp16_linear_fwd
 * (exact int64), then y[b][oc] = float(p64[b][oc]) * 2^(*d_exp_x + *d_exp_w)
 * (p64 rounded to float to nearest even, then scaled). y: float [B][OC];
 * d_max: device uint64 scratch (max |p64|). Workspace as ito_dfp16_linear_fwd. */
int ito_dfp16_linear_fwd_f32(const int16_t *x, const int32_t *d_exp_x, const int16_t *W, const int32_t *d_exp_w,
                             int B, int IC, int OC, void *workspace, size_t workspace_bytes, int64_t *p64,
                             uint64_t *d_max, float *y, void *stream);

/* DFP16 Linear forward with an FP32 output by the page's partial-accumulation
 * scheme ("Mixed Precision Training of Convolutional Neural Networks using
 * Integer Operations", section 4, "Handling overflows": INT16 products overflow
 * an INT32 accumulator after a few terms, so the kernels keep the accumulation
 * chains short and shift the inputs by one bit, convert each chain's INT32
 * partial to FP32, scale it by 2^(E_inp + E_wt) and accumulate it in FP32):
 *   x'  = input_shift ? round-half-up(x / 2) : x,  E_inp = *d_exp_x + input_shift
 *   for each chain j of `chain` consecutive ic (the last one shorter):
 *     p_j = (sum over the chain of x'[b][ic] * W[oc][ic]) modulo 2^32, as a
 *           two's-complement INT32 accumulator holds it
 *     t_j = float(float(p_j) * 2^(E_inp + *d_exp_w))  (to nearest even; the
 *           scaling itself is exact)
 *   y[b][oc] = (((0 + t_0) + t_1) + ...) with every addition rounded to float.
 * The page fixes no chain length: chain is a multiple of 64 in [64, 512]. A
 * chain whose sum leaves int32 wraps, as the page's hardware would; the
 * one-bit shift makes that impossible for chains of up to 3 terms and rare in
 * practice. x: int16 [B][IC] with exponent *d_exp_x; W: int16 [OC][IC] with
 * *d_exp_w; y: float [B][OC]. Workspace as ito_dfp16_linear_fwd. Exponents
 * outside int8 raise ITO_ERR_EXPONENT in the device error word.
 * Errors: ITO_ERR_ARG (NULL pointer, bad chain or input_shift, workspace),
 * ITO_ERR_SHAPE. */
int ito_dfp16_linear_fwd_f32_chained(const int16_t *x, const int32_t *d_exp_x, const int16_t *W,
                                     const int32_t *d_exp_w, int B, int IC, int OC, int32_t chain,
                                     int32_t input_shift, void *workspace, size_t workspace_bytes, float *y,
                                     void *stream);

/* Blocked-DFP ("Mixed Precision Training of Convolutional Neural Networks
 * using Integer Operations", section 3: Blocked-DFP raises the effective
 * range with several fine-grained exponents per tensor; the page gives no
 * block shape). Reading: each row of a [rows][cols] tensor is cut into blocks
 * of `block` consecutive elements (the last one shorter when block does not
 * divide cols), and each block is a DFP-16 tensor of its own with a signed
 * 8-bit exponent, converted as ito_dfp16_from_float converts a tensor.
 * mant: int16 [rows][cols]; exps: int8 [rows][ceil(cols / block)].
 * A block exponent outside int8 sets ITO_ERR_EXPONENT in the device error
 * word (the stored exponent is clamped), a non-finite input ITO_ERR_ARG.
 * Errors: ITO_ERR_ARG (NULL pointer), ITO_ERR_SHAPE (a size < 1). */
int ito_bdfp16_from_float(const float *f, int64_t rows, int64_t cols, int32_t block, int16_t *mant, int8_t *exps,
                          void *stream);
/* f = mant * 2^exp of its block (rounded once to float). */
int ito_bdfp16_to_float(const int16_t *mant, const int8_t *exps, int64_t rows, int64_t cols, int32_t block, float *f,
                        void *stream);

/* Linear forward with FP32 output over Blocked-DFP operands blocked along the
 * contraction with the same block length (section 4: the kernels produce FP32
 * outputs from DFP operands):
 *   y[b][oc] = float( sum over blocks j, in order, in double, of
 *                     P_j * 2^(ex[b][j] + ew[oc][j]) ),  P_j = sum_{k in block j} x[b][k] * W[oc][k]
 * P_j is exact (int64 via the limb contraction, one block per exact chunk) and
 * each term is exact in double; the result is deterministic.
 * x: int16 [B][IC]; ex: int8 [B][nb]; W: int16 [OC][IC]; ew: int8 [OC][nb];
 * nb = ceil(IC / block); block: a multiple of 64 in [64, 512]; y: float [B][OC].
 * Workspace: ito_dfp16_workspace_size(B, IC, OC) bytes, 256-byte aligned.
 * Errors: ITO_ERR_ARG (NULL pointer, workspace, block), ITO_ERR_SHAPE. */
int ito_bdfp16_linear_fwd_f32(const int16_t *x, const int8_t *ex, const int16_t *W, const int8_t *ew, int B, int IC,
                              int OC, int32_t block, void *workspace, size_t workspace_bytes, float *y, void *stream);

typedef struct ito_dfp16_model ito_dfp16_model;

/* A stack of DFP16 Linear layers dims[0] -> dims[1] -> ... -> dims[n_layers]
 * (no ReLU), every layer's weights 16-bit mantissas with exponent exp_w
 * (changed per layer only by the precision calls below), integer SGD rate
 * 2^-eta on the batch-summed gradient. Owns all its device memory. */
int ito_dfp16_model_create(const int32_t *dims, int n_layers, int batch, int32_t exp_w, int32_t eta,
                           ito_dfp16_model **out);
int ito_dfp16_model_destroy(ito_dfp16_model *m);
/* W: int16 [OC][IC] mantissas at the layer's current precision and exponent,
 * host (on_host != 0) or device memory. */
int ito_dfp16_model_set_weights(ito_dfp16_model *m, int layer, const int16_t *W, int on_host,
                                void *stream);
/* Named device tensors of the last step: "x", "p<l>" int64, "y<l>", "e<l>",
 * "pd<l>" int64, "pg<l>" int64, "g<l>", "w<l>" (int16 unless stated). */
int ito_dfp16_model_tensor(const ito_dfp16_model *m, const char *name, void **dev_ptr, int *elem_bytes,
                           int64_t *numel);
/* Scalars of the last step ("ey<l>", "ee<l>", "rs<l>", "rsd<l>", "rsg<l>",
 * "eg<l>", "k<l>", "nz<l>", "pmax<l>", "pdmax<l>", "pgmax<l>", "gabs<l>" =
 * sum |g<l>| (kept by the weight-gradient down-conversion)), copied to
 * host_out (n >= ito_dfp16_model_num_stats) at ito_dfp16_model_stat_index;
 * synchronises the device. */
int ito_dfp16_model_num_stats(const ito_dfp16_model *m);
int ito_dfp16_model_stat_index(const ito_dfp16_model *m, const char *name);
int ito_dfp16_model_read_stats(const ito_dfp16_model *m, int64_t *host_out, int n);
/* One training step: forward (each layer down-converted), top error = the
 * output (MSE against a zero target), then per layer from the top: delta
 * propagation with the pre-update weights (not the first layer), weight
 * gradient, update (saturated to the layer's precision). x: int16
 * [batch][dims[0]] with exponent exp_x. */
int ito_dfp16_train_step(ito_dfp16_model *m, const int16_t *x, int32_t exp_x, void *stream);

/* The DFP16 training step (ito_dfp16_train_step; "Mixed Precision Training of Convolutional
 * Neural Networks using Integer Operations", section 3) from a host buffer without waiting,
 * for a pipeline of steps: x_host (int16
 * mantissas [batch][in], exponent exp_x) is copied on a model-owned copy stream into one of
 * two model-owned device input buffers (alternating from call to call, after the step that
 * last read that buffer), the step runs on `stream` after the copy, and the statistics, in
 * the layout of ito_dfp16_model_read_stats (ito_dfp16_model_num_stats int64), are copied to
 * stats_host (may be NULL) on `stream`. The copy of the next call's batch overlaps this
 * step. Host buffers should be pinned; x_host must not change until `stream` has passed
 * this step. Errors: ITO_ERR_ARG, ITO_ERR_EXPONENT, ITO_ERR_CUDA. */
int ito_dfp16_train_step_host_async(ito_dfp16_model *m, const int16_t *x_host, int32_t exp_x,
                                    int64_t *stats_host, void *stream);

/* ------------------------------------------------------------------------
 * Adaptive precision training on the DFP16 model ("Adaptive Precision
 * Training for Resource Constrained Devices", section III: the Gavg metric of
 * Equation 4, Algorithm 1 (precision adjustment), Algorithm 2 (metric
 * evaluations inside an epoch, adjustment between epochs)).
 *
 * Representation (the page gives the formulas of epsilon and Gavg only as
 * missing images; this is the reading): each layer's weights are bits-bit
 * two's-complement mantissas, |W| <= 2^(bits-1) - 1, with one shared exponent
 * E_W, so the minimum resolution is epsilon = 2^E_W. The update saturates to
 * that range. Gavg of a layer = mean |g| / epsilon with g the batch-mean
 * weight gradient: sum|G| * 2^(E_G - E_W) / (N * B) for the batch-summed DFP
 * gradient G with exponent E_G, N weights and batch B (no learning rate, as
 * the page specifies), computed in double from the exact integer sum.
 * ---------------------------------------------------------------------- */

typedef struct ito_apt_params {
    int32_t k_init;      /* precision the weights start at (the page uses 6) */
    int32_t k_min;       /* precision limits, 2 <= k_min <= k_init <= k_max <= 16 */
    int32_t k_max;
    int32_t eval_every;  /* Gavg is evaluated at steps 0, eval_every, 2*eval_every, ... of an epoch */
    double t_min;        /* Algorithm 1: one more bit when Gavg < t_min ... */
    double t_max;        /* ... one bit less when Gavg > t_max (may be +infinity) */
} ito_apt_params;

/* A layer's weight precision and exponent (host values; no synchronisation). */
int ito_dfp16_model_get_precision(const ito_dfp16_model *m, int layer, int32_t *bits, int32_t *exp_w);

/* Change a layer's weight precision to `bits` (2..16): d = bits - current;
 * d > 0: W <- W * 2^d, E_W <- E_W - d (exact); d < 0: W <- clamp(rhu(W, -d),
 * +-(2^(bits-1) - 1)), E_W <- E_W - d. Enqueued on `stream`.
 * Errors: ITO_ERR_ARG, ITO_ERR_EXPONENT (E_W would leave int8). */
int ito_dfp16_model_set_precision(ito_dfp16_model *m, int layer, int32_t bits, void *stream);

/* Enable APT: every layer is set to p->k_init bits (ito_dfp16_model_set_precision)
 * and the step counter of the epoch is reset. From then on every
 * eval_every-th ito_dfp16_train_step of an epoch logs each layer's sum |G|
 * and E_G on the device (at most 256 evaluations per epoch).
 * Errors: ITO_ERR_ARG (parameters out of range), ITO_ERR_EXPONENT. */
int ito_dfp16_model_apt_enable(ito_dfp16_model *m, const ito_apt_params *p, void *stream);

/* End of an epoch (Algorithm 2): synchronises `stream`, computes each layer's
 * Gavg for every logged evaluation and their mean (in evaluation order), and
 * applies Algorithm 1: bits + 1 if mean < t_min and bits < k_max, else bits - 1
 * if mean > t_max and bits > k_min. Writes the means to gavg[n_layers] and the
 * new precisions to bits[n_layers] (either may be NULL) and starts a new epoch.
 * Errors: ITO_ERR_ARG (APT not enabled, or no evaluation logged), ITO_ERR_CUDA,
 * ITO_ERR_EXPONENT. */
int ito_dfp16_model_apt_epoch_end(ito_dfp16_model *m, double *gavg, int32_t *bits, void *stream);

/* Single-tensor forms: the DFP update of ito_dfp16_update with the result
 * saturated to +-(2^(bits-1) - 1) (2 <= bits <= 16; bits = 16 is ito_dfp16_update),
 * and the precision change of ito_dfp16_model_set_precision on an int16
 * tensor of n mantissas (the caller adjusts its exponent by bits_old - bits_new).
 * Errors: ITO_ERR_ARG (NULL pointer or bits out of range), ITO_ERR_SHAPE (n < 1). */
int ito_dfp16_update_bits(int16_t *W, const int16_t *g, const int32_t *d_exp_g, int64_t n, int32_t exp_w,
                          int32_t eta, int32_t bits, int32_t *d_k, uint32_t *d_nonzero, void *stream);
int ito_dfp_set_bits(int16_t *W, int64_t n, int32_t bits_old, int32_t bits_new, void *stream);

/* ------------------------------------------------------------------------
 * Measurement hooks (no counterpart in the pages; used by the benchmark)
 * ---------------------------------------------------------------------- */

typedef enum ito_prof_class {
    ITO_PROF_GEMM = 0,      /* tensor-core contractions; work = 2*M*N*K integer ops */
    ITO_PROF_REQUANT = 1,   /* requantisation passes; work = algorithmic HBM bytes */
    ITO_PROF_UPDATE = 2,    /* NITI weight updates; work = algorithmic HBM bytes */
    ITO_PROF_OTHER = 3,     /* conversion, im2col/col2im, pooling, top error; work = bytes */
    ITO_PROF_NCLASS = 4
} ito_prof_class;

/* Enables (1) or disables (0) per-kernel timing: when enabled, every kernel a
 * step launches is bracketed by CUDA events recorded on the step's stream
 * (inside the graph when steps replay from CUDA graphs). Synchronises the
 * device and frees captured graphs. */
int ito_model_profile(ito_model *m, int enable);

/* Adds up the timings of all steps since the last read (waiting for their
 * events) and clears them: ms[c], work[c] and launches[c] for each of the
 * ITO_PROF_NCLASS classes (arrays of ITO_PROF_NCLASS entries). Steps replayed
 * from a graph reuse its events, so with graphs only the last replay is held:
 * read after every step. */
int ito_model_profile_read(ito_model *m, double *ms, double *work, int64_t *launches);

/* Number of kernels the model launches per training step. */
int ito_model_kernels_per_step(const ito_model *m);

/* Measurement (no counterpart in the pages). Per-kernel timing of the DFP16 model, as
 * ito_model_profile /
 * ito_model_profile_read: an event pair on the launch's stream around every
 * launch of a step; classes ITO_PROF_GEMM (limb contractions; work = executed
 * bf16 operations, 8*M*N*K: four limb products per int16 multiply-add),
 * ITO_PROF_REQUANT (down-conversions; work = algorithmic HBM bytes),
 * ITO_PROF_UPDATE (weight updates; bytes) and ITO_PROF_OTHER. The model
 * launches directly (no graphs), so every step's events are kept until read.
 * Enabling synchronises the device. Errors: ITO_ERR_ARG, ITO_ERR_CUDA. */
int ito_dfp16_model_profile(ito_dfp16_model *m, int enable);
int ito_dfp16_model_profile_read(ito_dfp16_model *m, double *ms, double *work, int64_t *launches);

/* Number of kernels the DFP16 model launched in its last training step. */
int ito_dfp16_model_kernels_per_step(const ito_dfp16_model *m);

#ifdef __cplusplus
}
#endif

#endif /* ITO_H */
