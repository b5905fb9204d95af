/*
 * conv.h -- C ABI of libconv: the forward 2-D convolution (ONNX Conv
 * semantics) on one NVIDIA GB300 (sm_103a).
 *
 * The operation ("Convolution, pooling and resize", Layout and operands;
 * "Convolutions", sections 2.1 and 3):
 *
 *   Ho = floor((H + pad_top + pad_bottom - dil_h*(kh-1) - 1) / stride_h) + 1
 *   Wo = floor((W + pad_left + pad_right - dil_w*(kw-1) - 1) / stride_w) + 1
 *   y[n,co,oh,ow] = act( ( sum_{c,u,v} x[n, g*Cin/G + c, oh*sh - pt + u*dh,
 *                                                 ow*sw - pl + v*dw] * w[co,c,u,v] )
 *                        + bias[co] + residual[n,co,oh,ow] )
 *   with g = co / (Cout/G), zero outside the image, and the epilogue applied
 *   in that order -- sum, bias, residual, activation -- each step rounded to
 *   float32, the result rounded once to the element type (nearest even).
 *
 * Layouts: x is NCHW [n][c_in][h][w], w is OIHW [c_out][c_in/groups][kh][kw],
 * bias is [c_out], residual and y are NCHW [n][c_out][Ho][Wo]; all dense and
 * contiguous.  A one-dimensional convolution is h = 1 (with kh = 1).
 * One element type covers every operand; sums accumulate in float32.
 *
 * Ownership: every pointer is caller-owned memory.  conv_forward takes device
 * pointers; the library allocates nothing per call (it keeps a small
 * per-device cache of device attributes).  Pointers from a CUDA allocator
 * (256-byte aligned) take every fast path; other alignments are legal and
 * may run a slower variant of the same kernels.
 *
 * Asynchrony: conv_forward only enqueues kernels on `stream` (a cudaStream_t;
 * NULL is the legacy default stream) and returns; it never synchronises and
 * copies nothing to the host.  Results are bit-identical from run to run on
 * one device: no kernel uses atomics, and every sum has a fixed order.
 *
 * Errors: every function returns a conv_status.  Validation runs on the host
 * before anything is enqueued, so a call that returns an error other than
 * CONV_ERR_CUDA enqueued nothing.
 */
#ifndef CONV_GB300_H
#define CONV_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CONV_ABI_VERSION 1

#if defined(__GNUC__)
#define CONV_API __attribute__((visibility("default")))
#else
#define CONV_API
#endif

typedef enum conv_dtype {
  CONV_F32 = 0,  /* float32 operands and output                             */
  CONV_F16 = 1,  /* IEEE binary16 operands and output, float32 accumulation */
  CONV_BF16 = 2  /* bfloat16 operands and output, float32 accumulation      */
} conv_dtype;

/* Activations fused into the store ("Convolution, pooling and resize",
 * Layout and operands), with the ONNX operator definitions:
 *   relu max(t,0); sigmoid 1/(1+exp(-t)); tanh; silu t*sigmoid(t);
 *   hard_sigmoid max(0,min(1, alpha*t + beta));
 *   hard_swish t*max(0,min(1, t/6 + 1/2))   (alpha, beta unused);
 *   clip min(max(t, alpha), beta)            (alpha = min, beta = max);
 *   leaky_relu t >= 0 ? t : alpha*t. */
typedef enum conv_act {
  CONV_ACT_IDENTITY = 0,
  CONV_ACT_RELU = 1,
  CONV_ACT_SILU = 2,
  CONV_ACT_SIGMOID = 3,
  CONV_ACT_TANH = 4,
  CONV_ACT_HARD_SWISH = 5,
  CONV_ACT_HARD_SIGMOID = 6,
  CONV_ACT_CLIP = 7,
  CONV_ACT_LEAKY_RELU = 8
} conv_act;

/* conv_problem.flags: testing and measurement switches.  0 = automatic. */
#define CONV_FLAG_FORCE_FFMA 0x1u   /* the CUDA-core implicit GEMM for every shape   */
#define CONV_FLAG_NO_SPLIT_K 0x2u   /* never split k                                 */
#define CONV_FLAG_NO_WINDOW 0x4u    /* never the shifted-window tcgen05 variant       */
#define CONV_FLAG_NO_UNFOLD 0x8u    /* CUDA-core kernel: never the unfolded-input pre-pass */
#define CONV_FLAG_FORCE_UNFOLD 0x10u /* CUDA-core kernel: the unfolded-input pre-pass
                                        wherever it applies (output width a multiple of 4) */
#define CONV_FLAG_WINOGRAD 0x20u     /* Winograd F(2x2,3x3) wherever it applies (float32,
                                        3x3, stride 1, dilation 1, one group)      */
#define CONV_FLAG_NO_WINOGRAD 0x40u  /* never Winograd                                 */
#define CONV_FLAG_NO_DW_MMA 0x80u    /* 16-bit depthwise: the CUDA-core kernels, not the
                                        tensor-core band-matrix kernel              */
#define CONV_FLAG_NO_PW_MMA 0x4000u  /* 16-bit 1x1 layers: not the pointwise tensor-core
                                        tile kernel                                 */
#define CONV_FLAG_NO_CLUSTER_K 0x8000u /* split k: the ranges' float32 planes in scratch and a
                                        second kernel that adds them, not the reduction
                                        within a thread-block cluster               */
#define CONV_FLAG_SPLIT_K_SHIFT 8   /* bits 8..13: force this many ranges of k (1-63) */
#define CONV_FLAG_SPLIT_K_MASK 0x3f00u

/* The problem ("Convolution, pooling and resize", Layout and operands: a
 * problem struct with the shape, explicit pads, dilation, groups and the fused
 * activation).  Sizes are element counts. */
typedef struct conv_problem {
  int64_t n, c_in, h, w;            /* input NCHW                              */
  int64_t c_out, kh, kw;            /* weights OIHW [c_out][c_in/groups][kh][kw] */
  int64_t pad_top, pad_left, pad_bottom, pad_right; /* ONNX pads [t, l, b, r]  */
  int64_t stride_h, stride_w;       /* >= 1                                    */
  int64_t dil_h, dil_w;             /* >= 1                                    */
  int64_t groups;                   /* divides c_in and c_out                  */
  int32_t act;                      /* conv_act                                */
  float act_alpha, act_beta;        /* see conv_act                            */
  int32_t dtype;                    /* conv_dtype of x, w, bias, residual, y   */
  int32_t has_bias;                 /* bias pointer is read iff nonzero        */
  int32_t has_residual;             /* residual pointer is read iff nonzero    */
  uint32_t flags;                   /* CONV_FLAG_*                             */
} conv_problem;

typedef enum conv_status {
  CONV_OK = 0,
  CONV_ERR_SHAPE = 1,    /* a size < 1 (pads < 0), groups not dividing the
                            channels, no output position, or a size past a
                            kernel limit                                     */
  CONV_ERR_OVERFLOW = 2, /* an element count or offset overflows int64      */
  CONV_ERR_DTYPE = 3,    /* unknown conv_dtype                               */
  CONV_ERR_ACT = 4,      /* unknown conv_act                                 */
  CONV_ERR_NULL = 5,     /* a required pointer is NULL                       */
  CONV_ERR_SCRATCH = 6,  /* scratch smaller than conv_scratch_bytes reports  */
  CONV_ERR_ALIAS = 7,    /* y overlaps an input, or scratch overlaps an operand
                            ("Convolution, pooling and resize": scratch may
                            share a buffer with the operands only if its range
                            overlaps none of theirs)                          */
  CONV_ERR_DEVICE = 8,   /* no usable CUDA device, or not sm_103-class        */
  CONV_ERR_CUDA = 9,     /* a CUDA call or kernel launch failed               */
  CONV_ERR_ARG = 10      /* another invalid argument (e.g. a zero-length buffer) */
} conv_status;

/* What conv_forward runs for a problem ("Convolution, pooling and resize",
 * Variants: the variant a device runs is a function of the problem). */
typedef enum conv_variant {
  CONV_VARIANT_IGEMM_FFMA = 0,     /* implicit GEMM on CUDA cores, fused epilogue */
  CONV_VARIANT_IGEMM_FFMA_SPLIT = 1, /* the same with k split into ranges: the
                                      ranges of a tile are one thread-block
                                      cluster and add their float32 sums in
                                      range order through distributed shared
                                      memory, then the epilogue (one launch);
                                      or (CONV_FLAG_NO_CLUSTER_K, more than 16
                                      ranges, no such cluster on the device)
                                      each range into a float32 plane of
                                      scratch, then an ordered sum + epilogue
                                      pass; both give the same bits          */
  CONV_VARIANT_DEPTHWISE = 2,      /* direct halo-tiled kernel (one input channel
                                      per group, any channel multiplier)     */
  CONV_VARIANT_IGEMM_TC = 3,       /* implicit GEMM on tcgen05 tensor cores,
                                      input window gathered into shared memory */
  CONV_VARIANT_IGEMM_TC_WINDOW = 4, /* tcgen05 implicit GEMM over shifted windows of
                                      a zero-padded input band in shared memory
                                      (stride 1, or stride 2 split into 2x2
                                      phases; one group; the output's rows a
                                      multiple of 8 elements)                */
  CONV_VARIANT_WINOGRAD = 5,       /* Winograd F(2x2, 3x3) ("Convolutions",
                                      section 2.6): weight and input-tile
                                      transforms, sixteen products summed over
                                      channels on CUDA cores, output transform
                                      with the epilogue (float32, 3x3, stride
                                      1, dilation 1, one group; taken for 64 or
                                      more channels in and out)              */
  CONV_VARIANT_POINTWISE_MMA = 6   /* 16-bit 1x1 layers (stride 1, no padding, one
                                      group, Cin <= 256, Cout <= 64): tiles of
                                      output channels x 128 pixels on the tensor
                                      cores (warp-level mma.sync, float32 sums) */
} conv_variant;

/* The host-side plan of a problem for a device with `sm_count` SMs. */
typedef struct conv_plan_info {
  int32_t variant;        /* conv_variant                                     */
  int32_t split_k;        /* ranges of k (1 = the whole sum in one pass)       */
  int64_t ho, wo;         /* output size                                      */
  int64_t gemm_m;         /* output channels per group (Cout / groups)        */
  int64_t gemm_n;         /* output pixels (n * Ho * Wo)                      */
  int64_t gemm_k;         /* terms of each sum (Cin/groups * kh * kw)         */
  int64_t ctas;           /* thread blocks of the main kernel                 */
  int32_t tile_m, tile_n; /* output channels x pixels per thread block        */
  uint64_t scratch_bytes; /* device scratch conv_forward needs                */
} conv_plan_info;

/* ONNX Conv auto_pad values ("Convolution, pooling and resize", Layout and
 * operands: auto_pad is turned into explicit pads). */
typedef enum conv_auto_pad {
  CONV_AUTO_PAD_NOTSET = 0,      /* the explicit pads stay                          */
  CONV_AUTO_PAD_SAME_UPPER = 1,  /* Ho = ceil(H / stride); an odd pad's extra row /
                                    column at the end (bottom, right)               */
  CONV_AUTO_PAD_SAME_LOWER = 2,  /* the same, the extra row / column at the start   */
  CONV_AUTO_PAD_VALID = 3        /* no padding                                      */
} conv_auto_pad;

/* Library ABI version (CONV_ABI_VERSION). */
CONV_API int32_t conv_abi_version(void);

/* Human-readable name of a status code (static storage). */
CONV_API const char* conv_status_string(conv_status status);

/* Output size of `p` ("Convolutions", section 2.1, boxed equation, with the
 * two pads of an axis added separately).  Host only; validates `p` (all of
 * the checks of conv_forward that do not involve pointers).
 * Errors: CONV_ERR_NULL (p, ho or wo NULL), CONV_ERR_SHAPE, CONV_ERR_OVERFLOW,
 * CONV_ERR_DTYPE, CONV_ERR_ACT. */
CONV_API conv_status conv_output_shape(const conv_problem* p, int64_t* ho, int64_t* wo);

/* Writes into p's four pads what ONNX auto_pad `mode` prescribes for p's
 * input size, kernel, stride and dilation ("Convolution, pooling and resize",
 * Layout and operands).  For SAME_UPPER / SAME_LOWER the total padding of an
 * axis is max(0, (ceil(H/s) - 1)*s + d*(k-1) + 1 - H), split into halves, the
 * odd one at the end (UPPER) or the start (LOWER); VALID sets zeros; NOTSET
 * leaves the pads.  Host only.
 * Errors: CONV_ERR_NULL (p NULL), CONV_ERR_ARG (unknown mode), and the shape
 * checks of conv_output_shape on the result (p is not modified then). */
CONV_API conv_status conv_apply_auto_pad(conv_problem* p, int32_t mode);

/* The plan for a device with `sm_count` SMs: variant, k split, tile, grid and
 * scratch bytes.  Host only and a pure function of (p, sm_count), so split
 * decisions -- and with them the summation order -- depend only on the shape
 * and the device ("Convolution, pooling and resize", split k: the cut depends
 * only on the shape).  Assumes 256-byte aligned operands.
 * Errors: as conv_output_shape, and CONV_ERR_ARG for sm_count < 1. */
CONV_API conv_status conv_plan(const conv_problem* p, int32_t sm_count, conv_plan_info* out);

/* Scratch bytes conv_forward needs for `p` on the current CUDA device
 * ("Convolution, pooling and resize", Layout and operands: the scratch
 * query): the float32 partial planes of split k (ranges x output elements;
 * reported even where the ranges are reduced within a thread-block cluster,
 * which leaves them unused, so that a device where no such cluster fits can
 * still run the call),
 * the repacked weights of the shifted-window variant (channel tiles x k
 * blocks x tile channels x 16 bytes), the CUDA-core kernel's unfolded input
 * (float32, n x c_in x kw x padded rows x Wo) and transposed weights when it
 * uses them, 0 for the other variants.
 * Errors: as conv_plan, and CONV_ERR_DEVICE without a usable device. */
CONV_API conv_status conv_scratch_bytes(const conv_problem* p, size_t* bytes);

/* Scratch bytes conv_forward needs on the current device to run `p` one
 * image at a time ("Convolution, pooling and resize", Layout and operands: the
 * scratch query reports the whole batch and one image).  The CUDA-core
 * variant's split planes and unfolded input grow with the images it runs at
 * once: given less scratch than conv_scratch_bytes but at least this,
 * conv_forward runs the batch in chunks of as many whole images as fit, and
 * every output is computed by the same tile, k ranges and summation order as
 * in the whole-batch call -- the result is bit-identical.  The other variants'
 * scratch (repacked weights) does not depend on the batch: for them this
 * equals conv_scratch_bytes.
 * Errors: as conv_scratch_bytes. */
CONV_API conv_status conv_scratch_bytes_per_image(const conv_problem* p, size_t* bytes);

/* Writes a one-line description of what conv_forward runs for `p` on the
 * current device into buf (NUL-terminated, truncated to len), ending with
 * "launches=N", the number of kernels one conv_forward call launches
 * ("Convolution, pooling and resize", Variants: the library reports which
 * variant a problem runs). */
CONV_API conv_status conv_describe_variant(const conv_problem* p, char* buf, size_t len);

/* The same description for a device with `sm_count` SMs, on the host only
 * (no device is touched): the plan conv_plan makes for (p, sm_count), in
 * the words of conv_describe_variant.  Where the variant's choice depends on
 * the device beyond its SM count (whether a thread-block cluster of the k
 * ranges fits, checked when the call is launched) the description assumes
 * the sm_103 case.
 * Errors: CONV_ERR_NULL without buf or len, CONV_ERR_ARG for sm_count < 1,
 * the shape errors of conv_plan. */
CONV_API conv_status conv_describe_plan(const conv_problem* p, int32_t sm_count, char* buf, size_t len);

/* Enqueue y = conv(x, w) + bias + residual, activated, on `stream`.
 *   x, w, y     device pointers (required);
 *   bias        device pointer, read iff p->has_bias (then required);
 *   residual    device pointer, read iff p->has_residual (then required);
 *   scratch     device memory of scratch_bytes bytes, at least
 *               conv_scratch_bytes(p) -- or, for the CUDA-core variant, at
 *               least conv_scratch_bytes_per_image(p), which runs the batch in
 *               chunks of whole images with bit-identical results; may be
 *               NULL when that is 0.  The range conv_forward uses must overlap
 *               no operand; y must overlap no input.
 *   stream      cudaStream_t (NULL: legacy default stream).
 * Errors: those of conv_plan; CONV_ERR_NULL, CONV_ERR_SCRATCH, CONV_ERR_ALIAS
 * before anything is enqueued; CONV_ERR_DEVICE; CONV_ERR_CUDA when a launch
 * fails (the error is the launch's; nothing is synchronised). */
CONV_API conv_status conv_forward(const conv_problem* p, const void* x, const void* w,
                         const void* bias, const void* residual, void* y,
                         void* scratch, size_t scratch_bytes, void* stream);

/* Reads (and, if `reset`, clears) the current device's error word: nonzero
 * when a tensor-core kernel gave up a bounded wait (its output is then
 * incomplete); bits 0-15 come from the gather variant, bits 16-31 from the
 * shifted-window variant.  Synchronises the device; for tests and
 * diagnostics. */
CONV_API conv_status conv_device_error(uint32_t* word, int32_t reset);

/* Runs the tensor-core kernels' give-up path on its own, for tests: one block
 * allocates tensor memory, starts one 256-byte bulk copy, waits `limit_us`
 * microseconds (1 .. 100000) on an mbarrier that nothing arrives on, raises
 * its abort flag and reports into the shifted-window error word (bit 24 of
 * conv_device_error's word: the wait ran out; bit 25: the copy's drain ran
 * out), drains the copy, frees the tensor memory and returns.  The pages
 * describe no such call; it exists so that the bounded-wait mechanism the
 * kernels rely on can be checked without a failing convolution.
 * `report` (host, 5 words) receives: [0] waits that succeeded (0 expected),
 * [1] threads whose drain completed (64), [2] the abort flag (1), [3] 1 when
 * the block reached its end, [4] 1 when the copied bytes arrived intact.
 * Synchronous; uses the current device and allocates 528 bytes of device
 * memory for the call.  Errors: CONV_ERR_NULL, CONV_ERR_ARG (limit out of
 * range), CONV_ERR_DEVICE, CONV_ERR_CUDA. */
CONV_API conv_status conv_selftest_bounded_wait(uint32_t limit_us, uint32_t* report);

/* ---- ConvTranspose --------------------------------------------------------
 * The transposed convolution (ONNX ConvTranspose; "Convolution, pooling and
 * resize": weights [Cin][Cout/groups][kh][kw]; Variants: a Gemm of the
 * transposed weights with the input, then a gathering col2im with the same
 * epilogue):
 *
 *   Ho = stride_h*(H - 1) + out_pad_h + dil_h*(kh - 1) + 1 - pad_top - pad_bottom
 *   y[n,co,oh,ow] = act( sum_{c,u,v} x[n, g*Cin/G + c, (oh + pt - u*dh)/sh, (ow + pl - v*dw)/sw]
 *                                   * w[g*Cin/G + c, co - g*Cout/G, u, v]
 *                        + bias[co] + residual[n,co,oh,ow] )
 *
 * with g = co / (Cout/G) and only the terms whose divisions are exact and
 * land inside the input ("Convolutions", section 2.5: each input pixel
 * spreads the kernel over the output at s-strided positions).  The epilogue
 * and element types are those of conv_forward. */
typedef struct conv_transpose_problem {
  conv_problem conv;    /* n, c_in, h, w: the input; c_out: output channels;
                           kh, kw, pads, stride, dilation, groups, activation,
                           dtype, has_bias, has_residual as for conv_forward
                           (flags unused)                                     */
  int64_t out_pad_h, out_pad_w; /* ONNX output_padding, below max(stride, dilation) */
} conv_transpose_problem;

/* Output size of a transposed problem.  Host only.  Errors: CONV_ERR_NULL,
 * CONV_ERR_SHAPE (a size < 1, groups not dividing the channels, an
 * output_padding at or past max(stride, dilation), no output position, or a
 * size past a kernel limit), CONV_ERR_OVERFLOW, CONV_ERR_DTYPE, CONV_ERR_ACT. */
CONV_API conv_status conv_transpose_output_shape(const conv_transpose_problem* p, int64_t* ho, int64_t* wo);

/* Scratch bytes conv_transpose_forward needs on the current device: the
 * transposed weights, then the float32 Gemm result N x (Cout*kh*kw) x H*W. */
CONV_API conv_status conv_transpose_scratch_bytes(const conv_transpose_problem* p, size_t* bytes);

/* Enqueue the transposed convolution on `stream`; pointers as for
 * conv_forward (w laid out [c_in][c_out/groups][kh][kw]), scratch at least
 * conv_transpose_scratch_bytes, 256-byte aligned.  No atomics: the result
 * has the same bits on every run.  Errors: those of
 * conv_transpose_output_shape; CONV_ERR_NULL, CONV_ERR_SCRATCH,
 * CONV_ERR_ALIAS before anything is enqueued; CONV_ERR_DEVICE; CONV_ERR_CUDA. */
CONV_API conv_status conv_transpose_forward(const conv_transpose_problem* p, const void* x, const void* w,
                                            const void* bias, const void* residual, void* y, void* scratch,
                                            size_t scratch_bytes, void* stream);

/* ---- ConvInteger ----------------------------------------------------------
 * ONNX ConvInteger ("Convolution, pooling and resize", ConvInteger):
 *
 *   y[n,co,oh,ow] = sum_{c,u,v} (x[n, g*Cin/G + c, oh*sh - pt + u*dh, ow*sw - pl + v*dw] - x_zero)
 *                             * (w[co,c,u,v] - w_zero[co])
 *
 * in int32 with wrap-around (the exact sum modulo 2^32), with x and w each
 * uint8 or int8 in any mix; a tap outside the image is the quantized value
 * x_zero (the real value zero) and adds nothing.  The geometry is that of
 * conv_problem (pads, stride, dilation, groups; one-dimensional as h = 1);
 * act must be identity and has_bias / has_residual 0; dtype is ignored.
 * Layouts as for conv_forward (x NCHW, w OIHW, y NCHW int32). */
typedef enum conv_int_type {
  CONV_U8 = 0,  /* uint8, values 0..255 */
  CONV_I8 = 1   /* int8, two's complement, values -128..127 */
} conv_int_type;

/* Scratch bytes conv_integer_forward needs for p: the unfolded byte matrix
 * (groups x ceil(K/4) words x N*Ho*Wo pixels rounded to 4, K = Cin/G*kh*kw),
 * per-pixel and per-channel byte sums, and the weights as 4-byte words.
 * Host only.  Errors: those of conv_output_shape, CONV_ERR_DTYPE (x_type or
 * w_type not a conv_int_type), CONV_ERR_ARG (an activation, bias or residual
 * requested). */
CONV_API conv_status conv_integer_scratch_bytes(const conv_problem* p, int32_t x_type, int32_t w_type,
                                                size_t* bytes);

/* Enqueue ConvInteger on `stream`.
 *   x, w      device arrays of x_type / w_type elements (conv_int_type);
 *   x_zero    device pointer to one element of x_type;
 *   w_zero    device pointer to w_zero_count elements of w_type: 1 (one zero
 *             point) or c_out (one per output channel);
 *   y         device int32 array N x c_out x Ho x Wo;
 *   scratch   device memory of at least conv_integer_scratch_bytes, 256-byte
 *             aligned, overlapping no operand; y overlaps no input.
 * Results are exact and bit-identical across runs, devices and variants.
 * Errors: those of conv_integer_scratch_bytes; CONV_ERR_NULL, CONV_ERR_ARG
 * (w_zero_count), CONV_ERR_SCRATCH, CONV_ERR_ALIAS before anything is
 * enqueued; CONV_ERR_DEVICE; CONV_ERR_CUDA when a launch fails. */
CONV_API conv_status conv_integer_forward(const conv_problem* p, int32_t x_type, int32_t w_type,
                                          const void* x, const void* w, const void* x_zero,
                                          const void* w_zero, int32_t w_zero_count, int32_t* y,
                                          void* scratch, size_t scratch_bytes, void* stream);

/* Bytes of the library-owned scratch array of conv_forward_fixed_scratch. */
#define CONV_FIXED_SCRATCH_BYTES (8u << 20) /* 8 MiB */

/* conv_forward without caller-provided scratch, for callers that cannot
 * allocate device memory (no counterpart on the pages this library follows).
 *
 * Who needs it: code that may not call cudaMalloc -- a plug-in inside a host
 * framework that owns every device allocation, a latency-critical path that
 * must not enter the allocator, or a caller whose only CUDA code is this
 * library.  Such a caller still passes x, w, bias, residual and y (device
 * memory it was given), exactly as for conv_forward; the scratch conv_forward
 * would take from the caller -- the float32 planes of split k, the repacked
 * weights of the shifted-window tensor-core variant, the unfolded input and
 * transposed weights of the CUDA-core kernel, or Winograd's transformed
 * operands -- lives instead in one
 * fixed array of CONV_FIXED_SCRATCH_BYTES that the library declares in device
 * memory.  Every GPU that loads the library holds that array until the
 * process exits.
 *
 * When that scratch would exceed the array, the call runs the problem on a
 * variant that needs none, if there is one: the gather tensor-core kernel in
 * place of the shifted-window one, the direct CUDA-core kernel in place of
 * Winograd, the CUDA-core kernel gathering its input from x in place of the
 * unfolded copy, or k summed in one range in place of an automatic split.  Such a call gives results within the same error bound as
 * conv_forward's, but not necessarily the same bits (another summation order).
 *
 * Nothing is allocated by this call.  The first call on each device looks up
 * the array's device address (cudaGetSymbolAddress, with that device
 * current); make that first call before any stream capture on the device.
 * Every call shares the one array and leaves its last contents there (each
 * call overwrites every scratch byte it reads before reading it, so nothing
 * needs clearing); two calls whose kernels overlap on the GPU -- on different
 * streams, say -- race on it and must be serialised by the caller.
 *
 * Errors: those of conv_forward; CONV_ERR_SCRATCH when the problem's scratch
 * exceeds CONV_FIXED_SCRATCH_BYTES and no variant without scratch applies (a
 * split forced by the flags), before anything is enqueued; CONV_ERR_CUDA when
 * the array's address cannot be obtained. */
CONV_API conv_status conv_forward_fixed_scratch(const conv_problem* p, const void* x, const void* w,
                                                const void* bias, const void* residual, void* y,
                                                void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CONV_GB300_H */
