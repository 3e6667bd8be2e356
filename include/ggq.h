/*
 * ggq.h -- C ABI of the GB300 block-quantized dequantize + GEMV library.
 *
 * The library covers the hot path of GGUF local decode: read a GGUF v3 file,
 * copy its tensor payloads to device memory unchanged, and multiply
 * block-quantized weight matrices (Q8_0, Q4_K) by activation vectors with the
 * blocks decoded in registers.  Conventions follow the kernel list of the
 * culpeo.ws C++ engine blog, whose kernels never allocate and leave the output
 * memory to the caller: every compute entry point writes into
 * caller-provided device memory and enqueues its work on the caller's CUDA
 * stream without synchronising it.
 *
 * Shapes: a weight matrix has `rows` output features and `cols` input features
 * (GGUF ne0 = cols, stored fastest).  Row r is cols/32 consecutive 34-byte Q8_0
 * blocks, or cols/256 consecutive 144-byte Q4_K super-blocks.
 *
 * Return codes: 0 on success, a negative GGQ_E* code on failure (no partial
 * results are promised after a failure).  `ggq_strerror` names a code;
 * `ggq_last_error` gives a message for the last failure in the calling thread.
 *
 * Streams are passed as `void*` holding a cudaStream_t (NULL = legacy default).
 * Device pointers are plain `cudaMalloc`-style device addresses owned by the
 * caller unless stated otherwise.
 */
#ifndef GGQ_H
#define GGQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------- return codes */
#define GGQ_OK 0
#define GGQ_EINVAL (-1)    /* bad argument: NULL pointer, bad shape, M out of range, misaligned pointer */
#define GGQ_ETYPE (-2)     /* tensor type not supported by this operation */
#define GGQ_EIO (-3)       /* file could not be opened, mapped or read */
#define GGQ_EFORMAT (-4)   /* malformed GGUF: magic, version, truncation, offset, size overflow */
#define GGQ_ENOMEM (-5)    /* host or device allocation failed */
#define GGQ_ECUDA (-6)     /* a CUDA runtime call or kernel launch failed */
#define GGQ_ETIMEOUT (-7)  /* a kernel's bounded wait on its own copies ran out */
#define GGQ_ENOTFOUND (-8) /* no tensor / metadata key with that name */

/* ---------------------------------------------------- tensor type ids
 * F32 = 0 (the gguf_demo.py listing of "GGUF: The File Format...") and Q8_0 = 8
 * (the tensor-info example of "GGUF Inferencer in R" section 2.1) are on the
 * pages; F16, Q4_0, Q4_K and Q6_K use the ggml ids of real files. */
enum {
    GGQ_F32 = 0,
    GGQ_F16 = 1,
    GGQ_Q4_0 = 2,
    GGQ_Q8_0 = 8,
    GGQ_Q4_K = 12,
    GGQ_Q6_K = 14
};

/* GGUF metadata value types (GGUF v3): 4 = uint32, 8 = string, 9 = array are on
 * the pages; the others complete the v3 table. */
enum {
    GGQ_KV_U8 = 0, GGQ_KV_I8 = 1, GGQ_KV_U16 = 2, GGQ_KV_I16 = 3, GGQ_KV_U32 = 4,
    GGQ_KV_I32 = 5, GGQ_KV_F32 = 6, GGQ_KV_BOOL = 7, GGQ_KV_STRING = 8,
    GGQ_KV_ARRAY = 9, GGQ_KV_U64 = 10, GGQ_KV_I64 = 11, GGQ_KV_F64 = 12
};

/* ------------------------------------------------------------- loading */

typedef struct ggq_model ggq_model;

typedef struct {
    const char* name;  /* NUL-terminated; owned by the model */
    int32_t type;      /* GGQ_F32, GGQ_Q8_0, ... */
    int32_t n_dims;    /* 1..4 */
    int64_t ne[4];     /* extents, fastest first: ne[0] = cols; unused dims = 1 */
    uint64_t offset;   /* byte offset of the payload in the file's data blob */
    uint64_t nbytes;   /* payload size in bytes */
    const void* data;  /* device address of the payload (256-byte aligned), or NULL
                          for a model opened with GGQ_LOAD_METADATA_ONLY */
} ggq_tensor;

/* ggq_load_ex flags */
#define GGQ_LOAD_METADATA_ONLY 1u /* parse and validate; allocate no device memory */

/*
 * ggq_load -- read a GGUF v3 file and copy every tensor payload to the current
 * CUDA device, unchanged.
 *
 * The file is walked as "GGUF Inferencer in R" section 2.1 and "GGUF: The File
 * Format..." ("What is stored inside a GGUF file") lay it out: magic "GGUF",
 * uint32 version (3), uint64 tensor count, uint64 metadata count; typed
 * key/value entries (strings are uint64 length + bytes; unknown keys are
 * stepped over by their type); the tensor-info table (name, uint32 n_dims,
 * n_dims x uint64 extents, uint32 type, uint64 offset); padding to the next
 * multiple of 32; the data blob.  Offsets must be multiples of 32 and every
 * payload must lie inside the file.
 *
 * On success *out owns one device allocation holding all payloads (each at a
 * 256-byte-aligned address) plus host copies of names and metadata; release it
 * with ggq_free.  Errors: GGQ_EINVAL (NULL argument), GGQ_EIO, GGQ_EFORMAT,
 * GGQ_ETYPE (a tensor type whose payload size is unknown), GGQ_ENOMEM,
 * GGQ_ECUDA.  The copy is synchronous (the function returns after the data is
 * on the device).
 */
int ggq_load(const char* path, ggq_model** out);
int ggq_load_ex(const char* path, unsigned flags, ggq_model** out);

/* Same from a host buffer holding the file's bytes (not retained after return). */
int ggq_load_memory(const void* buf, size_t len, unsigned flags, ggq_model** out);

void ggq_free(ggq_model* model);

int ggq_version_of(const ggq_model* model, uint32_t* version);
int ggq_data_start(const ggq_model* model, uint64_t* offset);   /* file offset of the blob */
int ggq_num_tensors(const ggq_model* model, int64_t* n);
int ggq_tensor_info(const ggq_model* model, int64_t i, ggq_tensor* out);
int ggq_find_tensor(const ggq_model* model, const char* name, int64_t* i); /* GGQ_ENOTFOUND */

/*
 * Metadata access.  For scalar types *value points to the little-endian value
 * (value_bytes = its size); for strings to the bytes (not NUL-terminated;
 * value_bytes = length); for arrays to the raw encoded array starting at its
 * uint32 element type (value_bytes = encoded size).  Pointers stay valid until
 * ggq_free.
 */
int ggq_num_kv(const ggq_model* model, int64_t* n);
int ggq_kv_info(const ggq_model* model, int64_t i, const char** key, int32_t* vtype,
                const void** value, uint64_t* value_bytes);
int ggq_kv_find(const ggq_model* model, const char* key, int64_t* i); /* GGQ_ENOTFOUND */

/* ------------------------------------------------------------- compute */

/*
 * ggq_gemv -- y = W x for M activation rows, with W block-quantized.
 *
 *   y[m*rows + r] = sum_c w[r, c] * x[m*cols + c],   m < M, r < rows
 *
 * This is the matrix-vector kernel of the culpeo.ws kernel list (an r x c
 * weight times a c-vector gives an r-vector) and the product of the normalized
 * input with the transposed weight in "GGUF Inferencer in R" section 5.2, with the
 * weights decoded on the fly: Q8_0 w = d*q ("GGUF: The File Format...", "How
 * a Q8_0 block is stored"), Q4_K w = d*sc_j*q - dmin*m_j (the k-quant paragraph
 * of the same section; byte layout: fp16 d, fp16 dmin, 12 bytes of packed
 * 6-bit scales/mins, 128 bytes of nibbles), Q4_0 w = d*(u - 8) (the same
 * section: the Q8_0 layout with 4-bit integers, 18 bytes per 32 weights; byte
 * layout: fp16 d, then byte l holding the code u of weight l in its low nibble
 * and that of weight 16 + l in its high nibble), Q6_K w = d*sc[k/16]*(u - 32)
 * (the k-quant paragraph and the bits/weight loop of the same page, 210 bytes
 * per 256 weights; byte layout of real files: ql[128] low 4 bits, qh[64] high
 * 2 bits, 16 signed 8-bit sub-block scales, fp16 d; weight 128h + 32g + l has
 * the low bits in ql[64h + 32(g%2) + l] at bit 4(g/2) and the high bits in
 * qh[32h + l] at bit 2g), F32 the fp32 values as stored.  Decoded weights are
 * never written to memory; products accumulate in fp32 (any order).
 *
 *   type   GGQ_Q8_0 or GGQ_Q4_0 (cols % 32 == 0), GGQ_Q4_K or GGQ_Q6_K
 *          (cols % 256 == 0), GGQ_F32 (any cols >= 1)
 *   W      device, rows x row-bytes, row-major, 16-byte aligned
 *   x      device, fp32 [M, cols] row-major, 16-byte aligned
 *   y      device, fp32 [M, rows] row-major, 4-byte aligned; fully overwritten;
 *          must not overlap W or x (with 5..16 rows it may be zeroed first)
 *   M      1..16 (M > 1 is the small-batch variant: each decoded block is used
 *          for all M rows of x; from 5 rows on, Q8_0, Q4_K, Q4_0 and Q6_K
 *          (Q6_K with cols % 2048 == 0) run on the tensor cores in one pass
 *          over W; up to 4 rows, where the pre-scaled
 *          x of all M rows does not fit in shared memory, e.g. 4 rows of 14336
 *          columns, the rows run in groups, one pass over W per group)
 *   stream cudaStream_t
 *
 * Finite inputs with |x| < 2^70 are supported.  Errors: GGQ_EINVAL (NULL
 * pointer, rows outside 1..2^31-1, cols not a positive multiple of the block
 * or above 2^40, M outside 1..16, W not 16-byte aligned, x not 16-byte or y not
 * 4-byte aligned), GGQ_ETYPE (F16 or a type id not listed above), GGQ_ECUDA
 * (launch failure).  Asynchronous: returns after the launch.
 *
 * The call allocates no device memory and may be captured into a CUDA graph.
 * Calls on one stream run in stream order.
 */
int ggq_gemv(int type, const void* W, int64_t rows, int64_t cols, const float* x,
             float* y, int M, void* stream);

/*
 * ggq_gemv_multi -- ggq_gemv for n weight matrices of the same type and width
 * that share the activations x (the q, k and v projections of a layer, or its
 * gate and up projections), in one launch:
 *
 *   y[i][m*rows[i] + r] = sum_c w_i[r, c] * x[m*cols + c],   i < n
 *
 * W[i], rows[i], y[i] as for ggq_gemv; n in 1..4.  The rows of all n matrices
 * are spread evenly over the GPU as one list.  Same errors as ggq_gemv.
 * Asynchronous.
 */
int ggq_gemv_multi(int type, int n, const void* const* W, const int64_t* rows, int64_t cols,
                   const float* x, float* const* y, int M, void* stream);

/*
 * ggq_chain -- a fixed sequence of GEMV stages run by ONE kernel launch: the
 * weight-streaming part of a decode step ("GGUF Inferencer in R" section 4:
 * each generated token multiplies its activations by every weight matrix of
 * every layer, one matrix product after another).
 *
 * A stage is up to four matrices of the chain's type that share one x (as in
 * ggq_gemv_multi).  Stage s+1 starts reading its x only after every y of
 * stages 0..s has been written, so a stage's x may be an earlier stage's y.
 * Work that is not a GEMV between stages (norms, attention, activations) is
 * the caller's; a chain holds the GEMVs that follow one another directly.
 * Weights of later stages are streamed into shared memory while earlier
 * stages finish, so the chain keeps HBM busy across stage boundaries.
 *
 *   n        matrices in the stage, 1..4
 *   W[i]     device, rows[i] x row-bytes, 16-byte aligned
 *   rows[i]  1..2^31-1
 *   cols     multiple of 256, at most 2^20
 *   x        device fp32 [M, cols], 16-byte aligned
 *   y[i]     device fp32 [M, rows[i]], 4-byte aligned; fully overwritten
 */
typedef struct {
    int n;
    const void* W[4];
    int64_t rows[4];
    int64_t cols;
    const float* x;
    float* y[4];
} ggq_chain_stage;

typedef struct ggq_chain ggq_chain;

/*
 * ggq_chain_create -- validate `nstages` stages (1..65536) of type GGQ_Q8_0,
 * GGQ_Q4_K, GGQ_Q4_0 or GGQ_Q6_K for M activation rows (1..4; Q4_K and Q4_0
 * stages need cols >= 768, Q6_K stages cols % 2048 == 0, so that every row of
 * 210-byte super-blocks starts on 16 bytes; the pre-scaled x of all M rows of
 * the widest stage must fit in shared memory: 2 rows of 14336 columns do, 4 do
 * not), encode their copy descriptors and
 * store them in device memory on the current device.  The pointers are bound
 * at creation: the chain reads and writes the same buffers on every run.  The
 * caller owns the returned chain and frees it with ggq_chain_free.  Errors:
 * GGQ_EINVAL (malformed stage, misaligned pointer, unsupported shape; the
 * message names the stage), GGQ_ETYPE, GGQ_ENOMEM, GGQ_ECUDA.  Synchronous.
 */
int ggq_chain_create(int type, int M, int nstages, const ggq_chain_stage* stages, ggq_chain** out);

/*
 * Element-wise steps fused into a chain stage.  "GGUF Inferencer in R" section
 * 4 walks a layer: the input is RMS-normalized ("Normalize Input", before the
 * q/k/v and again before the gate/up projections), the gate projection goes
 * through SiLU and multiplies the up projection ("Activate Weights", before
 * the down projection), and the o and down projections are added to the
 * layer's input ("Add to Input").  The C++ engine post (culpeo.ws) lists the
 * same steps as the kernels rmsnorm, silu_mul and add.  A chain applies them
 * while it reads a stage's x and while it stores its y: no launch and no
 * extra pass over memory of their own.
 *
 *   x_op     GGQ_X_PLAIN     the stage multiplies x as given;
 *            GGQ_X_RMSNORM   ... norm_w[k] * x[m,k] / sqrt(mean_k x[m,k]^2 + eps)
 *                            (norm_w: device fp32 [cols], 16-byte aligned;
 *                            eps finite, >= 0; the mean over the stage's cols);
 *            GGQ_X_SILU_MUL  ... silu(x[m,k]) * up[m,k], silu(v) = v / (1 + e^-v)
 *                            (up: device fp32 [M, cols], 16-byte aligned).
 *   res[i]   NULL, or device fp32 [M, rows[i]], 4-byte aligned:
 *            y[i] = W_i x' + res[i] (res[i] may be the stage's own y[i]: the
 *            add happens as y[i] is written, after res[i] was read).
 * x, norm_w, up and res are only read; each may be an output of an earlier
 * stage of the chain (it is read after that stage's outputs are written).
 * Arithmetic is fp32: the sum of squares, 1 / sqrt by the IEEE square root and
 * division, SiLU with expf and an IEEE division.
 */
enum { GGQ_X_PLAIN = 0, GGQ_X_RMSNORM = 1, GGQ_X_SILU_MUL = 2 };

typedef struct {
    int x_op;
    float eps;
    const float* norm_w;
    const float* up;
    const float* res[4];
} ggq_chain_ops;

/*
 * ggq_chain_create_ops -- ggq_chain_create with the fused steps of each stage:
 * ops[s] for stage s (ops may be NULL: no fused steps anywhere).  Errors as for
 * ggq_chain_create; a bad x_op, a missing or misaligned norm_w / up / res, or a
 * negative or non-finite eps is GGQ_EINVAL naming the stage.  Synchronous.
 */
int ggq_chain_create_ops(int type, int M, int nstages, const ggq_chain_stage* stages, const ggq_chain_ops* ops,
                         ggq_chain** out);

/*
 * ggq_chain_create_typed -- ggq_chain_create_ops with a weight type per stage:
 * types[s] (GGQ_Q8_0, GGQ_Q4_K, GGQ_Q4_0 or GGQ_Q6_K, each with the shape
 * limits above) for stage s.  Files mix types from layer to layer and within a
 * layer ("GGUF: The File Format Powering Local LLM Inference", "Understanding
 * quantization names like Q4_K_M": Q4_K_M keeps part of attn_v and ffn_down in
 * Q6_K), and this lets the whole decode pass of such a file run as one chain.
 * A chain whose stages are all of one type runs the same kernel as
 * ggq_chain_create_ops.  A chain may also mix GGQ_Q6_K with one other type,
 * GGQ_Q4_K or GGQ_Q4_0 (Q4_K_M and Q4_K_S files; Q4_0 files with a Q6_K output
 * head): it runs a kernel that decodes each stage by its type (copy ring slots
 * sized for the larger).  ops may be NULL.  Errors as for ggq_chain_create_ops;
 * GGQ_ETYPE (naming the stage) for a type outside the four or a mix outside
 * those two.  Synchronous.
 */
int ggq_chain_create_typed(int M, int nstages, const int* types, const ggq_chain_stage* stages,
                           const ggq_chain_ops* ops, ggq_chain** out);

/*
 * ggq_chain_run -- run every stage of the chain, in order, as one cooperative
 * launch (every CTA resident at once, one per SM) on `stream` (cudaStream_t)
 * on the device the chain was created on.  The chain's stage counter lives in
 * the chain and is back at zero after each run, so runs may be captured into
 * a CUDA graph and replayed; runs of one chain must not overlap each other
 * (other streams).  Stage-boundary waits are bounded: if one runs out, the
 * kernel records it and ggq_device_status reports GGQ_ETIMEOUT; then call
 * ggq_chain_reset before the next run.  Allocates nothing.  Asynchronous.
 */
int ggq_chain_run(const ggq_chain* chain, void* stream);

/* ggq_chain_reset -- after a run that timed out: zero the chain's stage
 * counter and clear the device status word of the chain's device (read
 * ggq_device_status first to learn what happened; while the status word is
 * set, every bounded wait on that device gives up after a few polls).  No run
 * may be pending on the device.  Synchronous. */
int ggq_chain_reset(ggq_chain* chain);

/* ggq_chain_free -- release a chain (NULL is ignored).  No run may be pending. */
void ggq_chain_free(ggq_chain* chain);

/*
 * ggq_gemv_noalloc -- ggq_gemv that allocates nothing.  (No counterpart on the
 * pages: it exists for callers that may not allocate device memory.)
 *
 * Callers that cannot allow any device allocation at call time -- a server
 * that hands all device memory to its own pool at start-up and treats a later
 * cudaMalloc as a failure, or a latency-critical loop in which cudaMalloc /
 * cudaFree (which may synchronise the device) must never run -- use this
 * entry point: it is guaranteed to run the row-partitioned kernel, which
 * needs no scratch memory (no output row is split between CTAs), and it calls
 * no cudaMalloc, cudaFree or other allocating routine.  Shapes that would need
 * another kernel fail instead of falling back.
 *
 * Arguments and result as for ggq_gemv, within these limits: type GGQ_Q8_0,
 * GGQ_Q4_K or GGQ_Q4_0 (the last two with cols >= 768) with cols a multiple of
 * 256, or GGQ_Q6_K with cols a multiple of 2048; M in 1..4, x' of one
 * activation row in shared memory (cols up to about 40000 at M = 1); other
 * shapes fail with
 * GGQ_EINVAL.  Calls may overlap on the GPU: they share no device memory.
 */
int ggq_gemv_noalloc(int type, const void* W, int64_t rows, int64_t cols, const float* x, float* y, int M,
                     void* stream);

/*
 * ggq_gemm_prefill -- Y = X W^T for a whole prompt (M activation rows),
 * "GGUF Inferencer in R" section 4 (prefill takes the whole prompt through each
 * weight matrix as one large matrix product).  Weight tiles are decoded to bf16
 * in shared memory (exact fp32 decode, then one rounding to bf16) and
 * multiplied on the tcgen05 tensor cores with fp32 accumulation.
 *
 *   type   GGQ_Q4_K or GGQ_Q8_0, cols % 256 == 0 for both
 *   W      device, rows x (cols/256*144) (Q4_K) or rows x (cols/32*34) (Q8_0)
 *          bytes, 16-byte aligned; rows % 128 == 0
 *   X      device, bf16 bit patterns [M, cols] row-major, 16-byte aligned
 *   Y      device, fp32 [M, rows] row-major; fully overwritten
 *   M      multiple of 128, 128..65536
 *
 * Errors: GGQ_EINVAL, GGQ_ETYPE, GGQ_ECUDA.  The kernel's waits on its own
 * copies (and, for a tile computed as two halves along K, on the other half)
 * are bounded; if one runs out the kernel records it and ggq_device_status
 * reports GGQ_ETIMEOUT.  Calls on one device must not run concurrently (they
 * share the halves' sync words); calls on one stream may follow each other.
 * Asynchronous.
 */
int ggq_gemm_prefill(int type, const void* W, int64_t rows, int64_t cols,
                     const uint16_t* X, float* Y, int M, void* stream);

/*
 * ggq_dequantize -- out[r*cols + c] = w[r, c] as fp32 (test and inspection
 * aid; the GEMV path never writes decoded weights).  Types GGQ_Q8_0, GGQ_Q4_K,
 * GGQ_Q4_0, GGQ_Q6_K (decoded as in ggq_gemv) and GGQ_F32 (a device-to-device
 * copy);
 * cols a multiple of the type's block.  W 16-byte aligned, out 4-byte
 * aligned.  Asynchronous.
 */
int ggq_dequantize(int type, const void* W, int64_t rows, int64_t cols, float* out,
                   void* stream);

/*
 * ggq_embed -- token embedding lookup ("GGUF Inferencer in R" section 4, "Input
 * Embedding": a token id selects one row of the embedding table; the C++
 * engine post's embed(table, token)).  out[i*cols + k] = w[ids[i], k] as fp32,
 * decoded exactly as ggq_dequantize does, for i < n.
 *   type   GGQ_Q8_0, GGQ_Q4_K, GGQ_Q4_0, GGQ_Q6_K (table 2-byte aligned) or GGQ_F32
 *          (4-byte aligned); table device [rows, cols] in the type's layout
 *   ids    device int32 [n], n in 1..65535; out device fp32 [n, cols], 4-byte aligned
 * An id outside [0, rows) gives a row of zeros, and the next ggq_device_status
 * returns GGQ_EINVAL.  Errors: GGQ_ETYPE, GGQ_EINVAL (NULL, shape, n,
 * alignment), GGQ_ECUDA.  Allocates nothing.  Asynchronous.
 */
int ggq_embed(int type, const void* table, int64_t rows, int64_t cols, const int32_t* ids, int n, float* out,
              void* stream);

/*
 * ggq_device_status -- synchronise the current device, then return GGQ_ETIMEOUT
 * if any kernel of this library recorded a bounded-wait timeout since the last
 * call (and clear the record), GGQ_EINVAL if ggq_embed met an id outside its
 * table, GGQ_ECUDA if the device reports an error, else GGQ_OK.  Outputs of the launch that timed out, and of launches made after it
 * before this call, are undefined; a chain that timed out needs
 * ggq_chain_reset.  When one wait of a multi-CTA kernel runs out, the kernel's
 * other waits end within about a millisecond each, so the launch finishes
 * promptly.
 */
int ggq_device_status(void);

/* --------------------------------------------------------------- misc */
const char* ggq_strerror(int code);
const char* ggq_last_error(void);   /* thread-local message of the last failure */
int ggq_abi_version(void);          /* 1 */

#ifdef __cplusplus
}
#endif

#endif /* GGQ_H */
