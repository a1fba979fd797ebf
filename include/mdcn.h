/*
 * mdcn.h — C ABI of the GB300 (sm_103a) modulated deformable convolution
 * (DCNv2) library, libmdcn.so: the forward pass, and its gradients.
 *
 * The operation is the one described in "TensorRT plugin walkthrough:
 * modulatedDeformConvPlugin" (trdm.cn):
 *   section 2  inputs x, offset, mask, weight, optional bias; one output;
 *              NCHW; output dims (x.d0, weight.d0, offset.d2, offset.d3);
 *   section 3  attributes stride, padding, dilation (int[2] each), group,
 *              deformable_group; stride, dilation >= 1, padding >= 0,
 *              group, deformable_group >= 1; all five required;
 *   section 4  every tensor has the type of x; float32 or float16 (this
 *              library adds bfloat16 with the same semantics); linear NCHW;
 *              offset/mask batch = x batch, mask spatial = offset spatial,
 *              bias length = weight.d0;
 *   section 5  y[n,o,ho,wo] = bias[o] + sum over input channels c of the
 *              group of o and taps (i,j) of
 *                weight[o, c_l, i, j] * mask[n, gd*K + k, ho, wo]
 *                  * bilinear(x[n, c], ho*sh - ph + i*dh + offset[n, gd*2K + 2k, ho, wo],
 *                                      wo*sw - pw + j*dw + offset[n, gd*2K + 2k + 1, ho, wo])
 *              with K = kh*kw, k = i*kw + j, gd = c / (Cin/deformable_group),
 *              c_l = c - group_of(o)*(Cin/group); bilinear() is 0 outside the
 *              open range (-1, H) x (-1, W) and reads 0 for corners outside
 *              the image.
 *
 * Conventions shared by every entry point:
 *   - Pointers named x, offset, mask, weight, bias, out and workspace are
 *     DEVICE pointers, owned and allocated by the caller; the library never
 *     allocates, frees or keeps them. They must be 16-byte aligned
 *     (MDCN_ERR_ALIGN otherwise). Tensors are dense (contiguous) NCHW.
 *   - A call that fails validation launches nothing and writes nothing.
 *   - Forward calls are asynchronous on the given stream (a cudaStream_t
 *     passed as void*; NULL is the legacy default stream). No host
 *     synchronisation happens inside them. A CUDA launch error is reported
 *     as MDCN_ERR_CUDA (see mdcn_last_cuda_error).
 *   - No C++ exception crosses this interface; every call returns a status.
 *   - A handle is immutable after mdcn_create and may be used from several
 *     threads at once; concurrent forwards must use distinct workspaces.
 *   - Per-device set-up (kernel attributes, the allocation-free entry
 *     point's scratch address, cuBLAS handles of the ablation and the
 *     backward) is done on the first call on each device and kept for the
 *     life of the process. cudaDeviceReset discards it on the GPU side, so
 *     do not call the library on a device after resetting it in the same
 *     process.
 */
#ifndef MDCN_H
#define MDCN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mdcn_status {
    MDCN_OK = 0,
    MDCN_ERR_NULL = 1,        /* a required pointer argument is NULL */
    MDCN_ERR_ATTR = 2,        /* an attribute is out of its section-3 range */
    MDCN_ERR_SHAPE = 3,       /* tensor dims break a section-2/4 binding */
    MDCN_ERR_DTYPE = 4,       /* unknown mdcn_dtype value */
    MDCN_ERR_ALIGN = 5,       /* a device pointer is not 16-byte aligned */
    MDCN_ERR_WORKSPACE = 6,   /* workspace_bytes below mdcn_workspace_size() */
    MDCN_ERR_ARCH = 7,        /* the current device is not compute capability 10.3 */
    MDCN_ERR_CUDA = 8,        /* a CUDA runtime call or launch failed */
    MDCN_ERR_TIMEOUT = 9,     /* a device-side pipeline wait gave up (mdcn_query_status) */
    MDCN_ERR_UNSUPPORTED = 10 /* valid input beyond this library's limits (e.g. a dim >= 2^31) */
} mdcn_status;

/* Element type shared by x, offset, mask, weight, bias and out (section 4). */
typedef enum mdcn_dtype {
    MDCN_F32 = 0,  /* float32; contraction as split-TF32 (3 tensor-core passes), fp32 accumulate */
    MDCN_F16 = 1,  /* float16; fp16 columns, fp32 accumulate */
    MDCN_BF16 = 2  /* bfloat16; bf16 columns, fp32 accumulate (not on the page: an extension) */
} mdcn_dtype;

/* The five required attributes of section 3, index 0 = height, 1 = width. */
typedef struct mdcn_attrs {
    int64_t stride[2];
    int64_t padding[2];
    int64_t dilation[2];
    int64_t group;
    int64_t deformable_group;
} mdcn_attrs;

/* Dims of the inputs exactly as the tensors have them (section 2). */
typedef struct mdcn_dims {
    int64_t x[4];      /* N, Cin, H, W */
    int64_t offset[4]; /* N, 2*deformable_group*kh*kw, Ho, Wo */
    int64_t mask[4];   /* N, deformable_group*kh*kw, Ho, Wo */
    int64_t weight[4]; /* Cout, Cin/group, kh, kw */
    int64_t bias;      /* Cout when a bias is given, 0 when there is none */
} mdcn_dims;

typedef struct mdcn_handle_* mdcn_handle;

/* Validates attrs (section 3 ranges) and returns a handle holding a copy of
 * them in *out. Errors: MDCN_ERR_NULL (attrs or out NULL), MDCN_ERR_ATTR.
 * On error *out is left unchanged. Host only; touches no GPU. */
mdcn_status mdcn_create(const mdcn_attrs* attrs, mdcn_handle* out);

/* Optional overrides of the fused kernel's automatic execution plan, for
 * benchmarking and tuning. Results are bitwise identical for every stages and
 * kgroups setting with the same a_operand; a_operand changes which channels
 * share each tensor-core K-step (the rounding of the fp32 sums), tile_mode and
 * max_ctas move the points where output tiles are split between CTAs, which
 * changes the order of some fp32 additions. A zero (or -1 for tile_mode)
 * keeps the automatic choice. */
typedef struct mdcn_tuning {
    int32_t stages;    /* pipeline stages: 2, 4, 6 or 8 (0: automatic) */
    int32_t tile_mode; /* pixel tile: 0 = 128 consecutive pixels of N*Ho*Wo, 1 = 8x16 block of one image,
                          -1 = automatic */
    int32_t max_ctas;  /* cap on persistent CTAs (0: one per SM) */
    int32_t kgroups;   /* k-tiles the gather warps produce at once: 1, 2 or 4, dividing the stage count
                          (0: automatic) */
    int32_t a_operand; /* where the modulated columns (the MMA's A operand) are staged: 1 = shared memory,
                          2 = tensor memory (float16/bfloat16 with kgroups 2 only; the accumulators and
                          32 columns per stage must fit the 512 tensor-memory columns, with one
                          accumulator if two do not fit), 0 = automatic (tensor memory wherever it
                          is allowed) */
    int32_t ntile;     /* most output channels one tile holds: a multiple of 16 up to 512 (0: automatic).
                          Narrower tiles gather each pixel's columns once per tile of its group */
    int32_t path;      /* 1 = the fused implicit-GEMM kernel on the tensor cores; 2 = the direct kernel
                          on the CUDA cores (one thread per output pixel and up to 16 groups, fp32
                          sums, x read in NCHW; groups of at most 32 output channels, the fp32
                          weights of a thread's groups within 96 KB);
                          0 = automatic: direct where (Cin/group) * (Cout/group) <= 16, e.g.
                          depthwise, where the implicit GEMM would pad each channel unit to a 128-byte
                          k-tile and each group's outputs to 16 MMA columns; for a depthwise layer
                          (one input and one output channel per group) with Cin and Cin/dg multiples
                          of 4 and at most 49 taps, its channels-last form: x copied to
                          [N*H*W + 1][Cin] in the workspace first, then each lane reads a sampling
                          point's corners for 4 channels at once (2 launches; the same fp32 sums in
                          the same order, so the same bits). Forcing path 2 keeps x in NCHW */
} mdcn_tuning;

/* mdcn_create with plan overrides (tuning may be NULL = automatic). Errors as
 * mdcn_create, plus MDCN_ERR_ATTR for an override out of range. A plan that
 * the overrides make impossible (e.g. too many stages for shared memory) is
 * reported by the later calls as MDCN_ERR_UNSUPPORTED. */
mdcn_status mdcn_create_tuned(const mdcn_attrs* attrs, const mdcn_tuning* tuning, mdcn_handle* out);

/* Frees the handle (NULL is accepted). Nothing else is freed. */
mdcn_status mdcn_destroy(mdcn_handle handle);

/* Output dims by the section-2 rule: out_dims = {x[0], weight[0], offset[2],
 * offset[3]}, after checking every section-2/4 binding: offset and mask batch
 * = x batch; mask spatial = offset spatial; offset channels =
 * 2*dg*kh*kw; mask channels = dg*kh*kw; weight.d1 = Cin/group with group
 * dividing Cin and Cout; dg dividing Cin; bias = Cout or 0; every dim >= 1.
 * Ho and Wo are NOT recomputed from the convolution formula. Host only.
 * Errors: MDCN_ERR_NULL, MDCN_ERR_SHAPE, MDCN_ERR_UNSUPPORTED (a dim or an
 * element count beyond 2^31-1 / 2^62). */
mdcn_status mdcn_output_dims(mdcn_handle handle, const mdcn_dims* dims, int64_t out_dims[4]);

/* Bytes of device workspace mdcn_forward needs for these dims and dtype
 * (a status word, the channels-last copy of x, the repacked weight, and the
 * fp32 partial sums of output tiles split between CTAs; a direct plan, see
 * mdcn_tuning.path, needs the 1 KB header only, plus x channels-last,
 * (N*H*W + 1) * Cin elements, for its depthwise channels-last form). Host
 * only. */
mdcn_status mdcn_workspace_size(mdcn_handle handle, const mdcn_dims* dims, mdcn_dtype dtype,
                                size_t* bytes);

/* The execution plan mdcn_forward would use for these dims and dtype on the
 * current device (needs a compute capability 10.3 device for its SM count). */
typedef struct mdcn_plan_info {
    int64_t tiles;          /* output tiles: 128 pixels x up to 256 output channels of one group */
    int64_t ktiles_per_tile; /* k-tiles (128 bytes of channels of one tap) of one tile */
    int64_t ktiles_per_cta; /* consecutive k-tiles each persistent CTA takes */
    int32_t ctas;           /* persistent CTAs of the fused kernel */
    int32_t split;          /* 1 when some tile is split between CTAs (summed inside the fused kernel) */
    int32_t stages, kgroups, tile_mode;
    int32_t launches;       /* kernels one mdcn_forward launches: prep (1, or 2 when x needs the staged
                               transpose) and the fused kernel; 1 for a direct plan, 2 for its
                               depthwise channels-last form */
    int32_t a_operand;      /* 1: A stages in shared memory, 2: in tensor memory (0: direct plan) */
    int32_t path;           /* 1: fused implicit GEMM, 2: direct kernel (the tile fields above are then 0) */
} mdcn_plan_info;

/* Errors as mdcn_workspace_size, plus MDCN_ERR_ARCH / MDCN_ERR_CUDA from the
 * device check. The source pages have no counterpart: this is a diagnostic. */
mdcn_status mdcn_query_plan(mdcn_handle handle, const mdcn_dims* dims, mdcn_dtype dtype, mdcn_plan_info* info);

/* The forward pass (section 5, steps 1-3) as one fused implicit-GEMM kernel:
 * producer warps compute each sampling point from offset and mask, gather
 * and modulate the columns straight into the tensor core's operand stages
 * (tensor memory, or shared memory where the plan keeps them there), tcgen05
 * tensor-core MMAs accumulate in tensor memory, the epilogue adds the bias
 * and writes NCHW. The im2col column matrix never reaches device memory.
 * Persistent CTAs (one per SM) take equal consecutive ranges of the k-tiles
 * of all output tiles (stream-K). A tile split between CTAs is finished by
 * the CTA holding its last k-tiles, which processes its ranges last to first
 * and so reaches it last: it adds the other CTAs' fp32 partial sums, in k
 * order, before its epilogue. One small kernel runs
 * first, into workspace: x to channels-last and the weight repack (two
 * launches for shapes whose transpose needs the staged kernel).
 *   x [N,Cin,H,W], offset [N,2*dg*kh*kw,Ho,Wo], mask [N,dg*kh*kw,Ho,Wo],
 *   weight [Cout,Cin/group,kh,kw], bias_or_null [Cout] or NULL,
 *   out [N,Cout,Ho,Wo] (written), workspace of workspace_bytes (scratch,
 *   contents undefined afterwards except the status word).
 * dims->bias must be 0 exactly when bias_or_null is NULL.
 * stream: cudaStream_t as void*. Requires a compute capability 10.3 device
 * current on the calling thread. */
mdcn_status mdcn_forward(mdcn_handle handle, const void* x, const void* offset, const void* mask,
                         const void* weight, const void* bias_or_null, void* out,
                         void* workspace, size_t workspace_bytes,
                         const mdcn_dims* dims, mdcn_dtype dtype, void* stream);

/* The three steps of mdcn_forward as separate calls, for callers that pack a
 * constant weight once or time the steps on their own. Same argument rules
 * and workspace as mdcn_forward; x and weight are read only by the step that
 * names them. Plans of the fused kernel only: for a direct plan (see
 * mdcn_tuning.path; mdcn_query_plan tells) each returns MDCN_ERR_UNSUPPORTED
 * and launches nothing. Run on one stream, with one workspace, and
 * mdcn_forward_prepared after the other two:
 *   mdcn_prepare_input:    x -> channels-last copy in workspace; clears the
 *                          workspace status word;
 *   mdcn_pack_weight:      weight -> packed K-major copy in workspace;
 *   mdcn_forward_prepared: the fused kernel (sampling from offset and mask,
 *                          section 5 step 1; gather; contraction; bias;
 *                          the sums of split tiles). */
mdcn_status mdcn_prepare_input(mdcn_handle handle, const void* x, void* workspace, size_t workspace_bytes,
                               const mdcn_dims* dims, mdcn_dtype dtype, void* stream);
mdcn_status mdcn_pack_weight(mdcn_handle handle, const void* weight, void* workspace, size_t workspace_bytes,
                             const mdcn_dims* dims, mdcn_dtype dtype, void* stream);
mdcn_status mdcn_forward_prepared(mdcn_handle handle, const void* offset, const void* mask, const void* bias_or_null,
                                  void* out, void* workspace, size_t workspace_bytes, const mdcn_dims* dims,
                                  mdcn_dtype dtype, void* stream);

/* The "pack" form of the layer: offset and mask computed from x by an
 * ordinary convolution in front of the deformable one, as mmcv's
 * ModulatedDeformConv2dPack does (the pages name the modulated deformable
 * convolution of mmcv but do not spell this front end out; the reading here:
 *   om     = conv2d(x, weight_om, bias_om) with the handle's stride, padding
 *            and dilation, group 1; weight_om [3*dg*kh*kw, Cin, kh, kw],
 *            bias_om [3*dg*kh*kw] (both required);
 *   offset = om[:, 0 : 2*dg*kh*kw]                 (written to offset_out);
 *   mask   = sigmoid(om[:, 2*dg*kh*kw : 3*dg*kh*kw]) (written to mask_out);
 *   out    = mdcn_forward(x, offset, mask, weight, bias_or_null).)
 * dims describes the deformable layer as for mdcn_forward; its offset and
 * mask dims (those of offset_out and mask_out) must have the convolution's
 * spatial size floor((H + 2p - d(k-1) - 1)/s) + 1, else MDCN_ERR_SHAPE. All
 * pointers are device pointers (16-byte aligned); the workspace is at least
 * mdcn_pack_workspace_size bytes. Asynchronous on the stream: the front end is
 * the fused kernel run as a plain convolution into the workspace, a small
 * kernel splits its output into offset_out and sigmoid(mask) in mask_out, then
 * the deformable convolution reads them (reusing the workspace's channels-last
 * x when its layout is the same). */
mdcn_status mdcn_pack_workspace_size(mdcn_handle handle, const mdcn_dims* dims, mdcn_dtype dtype, size_t* bytes);
mdcn_status mdcn_forward_pack(mdcn_handle handle, const void* x, const void* weight_om, const void* bias_om,
                              const void* weight, const void* bias_or_null, void* offset_out, void* mask_out,
                              void* out, void* workspace, size_t workspace_bytes, const mdcn_dims* dims,
                              mdcn_dtype dtype, void* stream);

/* Bytes of the device buffer that mdcn_forward_host needs for these dims
 * and dtype: room for the device copies of x, offset, mask, weight and bias,
 * the output, and the mdcn_forward workspace, each 256-byte aligned. Host
 * only. Errors as mdcn_workspace_size. */
mdcn_status mdcn_host_buffer_size(mdcn_handle handle, const mdcn_dims* dims, mdcn_dtype dtype, size_t* bytes);

/* The forward from and to HOST memory. The source pages have no counterpart:
 * this entry point is for callers whose tensors live on the host.
 *   x_host, offset_host, mask_host, weight_host, bias_host_or_null: host
 *   pointers to dense NCHW inputs (layouts and rules as mdcn_forward);
 *   out_host: host pointer receiving the NCHW output;
 *   device_buffer: caller-owned DEVICE memory of device_buffer_bytes >=
 *   mdcn_host_buffer_size, 16-byte aligned; it holds the device copies, the
 *   output and the workspace (contents undefined afterwards).
 * On the stream, in order: one cudaMemcpyAsync per input into device_buffer,
 * the kernels of mdcn_forward, one cudaMemcpyAsync of the output to out_host.
 * Asynchronous like every forward: the host buffers must stay valid and the
 * inputs unmodified, and out_host must not be read, until the stream has
 * passed the call. With page-locked host memory (cudaHostAlloc,
 * cudaHostRegister) the copies run on the copy engines and overlap the work of
 * other streams, so calls on two streams with two device buffers pipeline the
 * copies of one call with the kernels of the other; pageable memory works, but
 * its copies are staged through the driver. Everything is validated before
 * the first copy: a call that fails validation copies and launches nothing. */
mdcn_status mdcn_forward_host(mdcn_handle handle, const void* x_host, const void* offset_host, const void* mask_host,
                              const void* weight_host, const void* bias_host_or_null, void* out_host,
                              void* device_buffer, size_t device_buffer_bytes, const mdcn_dims* dims,
                              mdcn_dtype dtype, void* stream);

/* Workspace bytes for mdcn_forward_im2col_gemm (the column matrix of the
 * whole batch plus a float32 GEMM output). Host only. */
mdcn_status mdcn_im2col_gemm_workspace_size(mdcn_handle handle, const mdcn_dims* dims,
                                            mdcn_dtype dtype, size_t* bytes);

/* Ablation: the same forward as the page's own two-stage design, kept for
 * comparison only — a deformable im2col kernel writes the column matrix
 * [N][Cin*kh*kw][Ho*Wo] into workspace (in the I/O dtype), one strided-
 * batched cuBLAS GEMM per group contracts it with the weight (fp32
 * accumulate, no TF32) into a float32 buffer, and a third kernel adds the
 * bias and writes the output. Same arguments and rules as mdcn_forward. */
mdcn_status mdcn_forward_im2col_gemm(mdcn_handle handle, const void* x, const void* offset,
                                     const void* mask, const void* weight, const void* bias_or_null,
                                     void* out, void* workspace, size_t workspace_bytes,
                                     const mdcn_dims* dims, mdcn_dtype dtype, void* stream);

/* ---------------------------------------------------------------- backward
 * The gradients of L = sum(grad_out * y) for y = mdcn_forward(x, offset,
 * mask, weight, bias), for training. The page defines only the forward
 * (section 5 steps 1-3); this is the gradient of that definition, read as:
 * inside the open range (-1, H) x (-1, W) the sample is the bilinear
 * polynomial of the cell whose corner is (floor h, floor w) over the
 * zero-extended image, with that polynomial's slopes (the right-hand slope
 * where h or w is an integer); outside the range the sample and its slopes
 * are 0, as the forward's range test gives. With G[n,c,k,p] = sum over the
 * output channels o of c's group of weight[o,c_l,k] * grad_out[n,o,p]:
 *   grad_x[n,c,corner]          = sum of G * mask * corner weight
 *   grad_offset[n,gd*2K+2k(+1),p] = mask * sum over c of gd: G * dv/dh (dv/dw)
 *   grad_mask[n,gd*K+k,p]       = sum over c of gd: G * v
 *   grad_weight[o,c_l,k]        = sum over n, p: grad_out[n,o,p] * mask * v
 *   grad_bias[o]                = sum over n, p: grad_out[n,o,p]
 * (v = the bilinear sample of x[n,c] at the point of tap k, pixel p). */

/* Bytes of device workspace mdcn_backward needs (a status word, the
 * tap-major weight, an fp32 weight gradient, and per chunk of images:
 * channels-last x, an fp32 grad_x accumulator, the fp32 column gradients and
 * the modulated columns; chunks hold as many images as fit in about 256 MB of
 * these, at least one; then, where the contractions run on the tensor cores,
 * the fp32 slices of the split weight-gradient contraction, else, for group
 * 1, grad_out re-laid [Cout][n][Ho*Wo] and a 32 MB cuBLAS workspace).
 * Host only. Errors as mdcn_workspace_size. */
mdcn_status mdcn_backward_workspace_size(mdcn_handle handle, const mdcn_dims* dims, mdcn_dtype dtype, size_t* bytes);

/* Kernel launches, memsets and cuBLAS calls one mdcn_backward call makes for
 * these dims and dtype (a diagnostic; the page has no counterpart). Host only. */
mdcn_status mdcn_backward_launches(mdcn_handle handle, const mdcn_dims* dims, mdcn_dtype dtype, int32_t* launches);

/* The backward pass. Inputs (DEVICE pointers, dense NCHW, one dtype, as for
 * mdcn_forward): x [N,Cin,H,W], offset [N,2*dg*kh*kw,Ho,Wo], mask
 * [N,dg*kh*kw,Ho,Wo], weight [Cout,Cin/group,kh,kw], grad_out [N,Cout,Ho,Wo].
 * Outputs (written, same dtype and dims as the tensor they belong to):
 * grad_x, grad_offset, grad_mask, grad_weight, and grad_bias_or_null [Cout]
 * (NULL: not computed; dims->bias must be Cout exactly when it is given).
 * workspace: >= mdcn_backward_workspace_size bytes, contents undefined
 * afterwards; its first word is the call's device status word, which
 * mdcn_query_status reads (a bounded wait of the tensor-core GEMMs that gave
 * up sets it). Every pointer 16-byte aligned. Arithmetic in fp32: for
 * float16 and bfloat16 the two contractions (the column gradients W^T *
 * grad_out, and the weight gradient grad_out * columns^T) run on this
 * library's tcgen05 tensor-core GEMM with fp32 accumulation, where Ho*Wo and
 * (Cin/group)*kh*kw are multiples of 8 (TMA's 16-byte row rule), else, and
 * for float32 (fp32 products, no TF32), as cuBLAS GEMMs. grad_x is summed
 * with fp32 atomic additions, so its last bits may differ from run to run;
 * the other gradients are deterministic (the split weight-gradient
 * contraction is summed in a fixed order). Asynchronous on the stream; a call
 * that fails validation launches nothing and writes nothing.
 * Errors: MDCN_ERR_NULL, MDCN_ERR_SHAPE, MDCN_ERR_DTYPE, MDCN_ERR_ALIGN,
 * MDCN_ERR_WORKSPACE, MDCN_ERR_UNSUPPORTED (a GEMM dimension beyond 2^31-1,
 * or a coordinate beyond 2^24), MDCN_ERR_ARCH, MDCN_ERR_CUDA. */
mdcn_status mdcn_backward(mdcn_handle handle, const void* x, const void* offset, const void* mask, const void* weight,
                          const void* grad_out, void* grad_x, void* grad_offset, void* grad_mask, void* grad_weight,
                          void* grad_bias_or_null, void* workspace, size_t workspace_bytes, const mdcn_dims* dims,
                          mdcn_dtype dtype, void* stream);

/* mdcn_forward without a caller-supplied workspace, for callers that cannot
 * allocate device memory on their execution path (a serving loop that reserves
 * all memory at start-up, a runtime whose execute step must not call
 * cudaMalloc, or plain C code without a device allocator). The source pages
 * have no counterpart of this entry point.
 *   - Scratch: a fixed 64 MiB device array inside libmdcn.so, present on every
 *     GPU that loads the library until the process exits. Calls whose
 *     mdcn_workspace_size exceeds 64 MiB are rejected with MDCN_ERR_WORKSPACE
 *     before anything is launched.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - The first call on a device looks up the array's device address (one
 *     cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture.
 *   - Every call on a device shares the one array, which keeps the last call's
 *     contents; each call overwrites what it reads, and clears the status word.
 *     Calls that overlap on the GPU (other streams, other threads) race on the
 *     array and must be serialised by the caller.
 *   - Otherwise identical to mdcn_forward: same arguments (minus workspace),
 *     validation (the device is checked before the array's address is looked
 *     up, so a GPU of another architecture gets MDCN_ERR_ARCH), kernels and
 *     results. The device status word lives in the array:
 *     mdcn_noalloc_query_status reads it. */
mdcn_status mdcn_forward_noalloc(mdcn_handle handle, const void* x, const void* offset, const void* mask,
                                 const void* weight, const void* bias_or_null, void* out,
                                 const mdcn_dims* dims, mdcn_dtype dtype, void* stream);

/* mdcn_query_status for mdcn_forward_noalloc, whose callers never see the
 * fixed array's address: reads the status word that the last
 * mdcn_forward_noalloc on the current device left in the array (synchronising
 * the stream), stores its raw bits in *device_bits (may be NULL) and clears
 * it. Returns MDCN_ERR_TIMEOUT when a pipeline wait of that call gave up (its
 * output is then unspecified), MDCN_OK when the word is clear, MDCN_ERR_ARCH
 * on a device other than compute capability 10.3, MDCN_ERR_CUDA when a CUDA
 * call fails. Like the forward, it must not overlap a noalloc forward that is
 * still running on another stream. The source pages have no counterpart. */
mdcn_status mdcn_noalloc_query_status(void* stream, uint32_t* device_bits);

/* Reads the device status word that the last mdcn_forward on this workspace
 * left (synchronising the stream), stores its raw bits in *device_bits (may
 * be NULL) and clears it. Returns MDCN_ERR_TIMEOUT when a pipeline wait in
 * the fused kernel gave up (its output is then unspecified), MDCN_OK when
 * the word is clear, MDCN_ERR_CUDA when the copy fails. */
mdcn_status mdcn_query_status(const void* workspace, void* stream, uint32_t* device_bits);

/* Self-test of the bounded wait used by every pipeline wait of the fused
 * kernel: launches one block that waits on a shared-memory barrier that
 * nothing ever signals, with the given limit in microseconds (1..10^7),
 * then synchronises the stream. Returns MDCN_ERR_TIMEOUT when the wait gave
 * up as designed, MDCN_OK if it (wrongly) completed. The GPU stays usable.
 * status_word: a caller-owned device buffer of at least 16 bytes. */
mdcn_status mdcn_selftest_wait_timeout(void* status_word, uint32_t limit_us, void* stream);

/* cudaError_t value behind the last MDCN_ERR_CUDA returned on this thread. */
int mdcn_last_cuda_error(void);

/* Static description of a status code. Never NULL. */
const char* mdcn_status_string(mdcn_status status);

#ifdef __cplusplus
}
#endif

#endif /* MDCN_H */
