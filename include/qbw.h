/*
 * qbw.h -- block-quantized weight matrix-vector products for NVIDIA GB300
 * (sm_103a).  C ABI: plain pointers, sizes and an opaque CUDA stream.
 *
 * Weights are raw GGUF block bytes, exactly as a GGUF file stores them:
 *
 *   Q8_0 block, 34 bytes: fp16 scale d (little-endian), then 32 int8 codes q;
 *        weight = d * q.
 *   Q4_0 block, 18 bytes: fp16 scale d, then 16 bytes qs; code j (0..15) is the
 *        low nibble of qs[j], code j+16 the high nibble; weight = d * (code - 8).
 *
 * (gem docs/research/architecture.md, "M4 Max operating assumptions": Q4_0 is
 * the "32-element/18-byte block" the decode matrix-vector kernel streams, Q8_0
 * the token-table and quality-baseline format.  The nibble order is the GGUF
 * block_q4_0 record's.)
 *
 * A weight matrix W with N output rows and K inputs (K a multiple of 32) is N
 * rows of K/32 consecutive blocks, rows back to back with no padding: the
 * [out, in] row-major layout of a linear layer (SafeC Gemma 4 design notes,
 * "Math primitives implementation status").  Row n holds output n's weights.
 *
 * Activations are fp32 or bf16 (QBW_F32 / QBW_BF16); they are never quantized.
 * Products accumulate in fp32.
 *
 * Pointers.  Every w, x, y, out, X, Y, workspace pointer is a DEVICE pointer
 * (or managed memory) on the current CUDA device.  The caller owns every
 * buffer: the calls allocate nothing, free nothing and keep no pointer after
 * they return (qbw_chain_create is the one call that allocates).  Outputs
 * must not overlap inputs.
 *
 * Library state.  Loading the library on a device reserves, as static device
 * arrays of the library's module, besides a 4-byte fault word
 * (qbw_fault_read):
 *   - the split-tile scratch of the tensor-core M = 1 kernels (qmv_q4_0,
 *     qmv_gateup_q4_0, qmv_q4_k and qmv_mixbit at the sizes
 *     that take them, and qmm_q4_0_smallM with M <= 2): 32 slots of 160 CTAs x
 *     2 x 128 tagged 64-bit words, 10,485,760 bytes.  When a 128-row output
 *     tile is split between two CTAs, the CTA that does not write it publishes its partial
 *     sums there, each word tagged with its launch's grid identifier, and the
 *     CTA that writes the tile takes only words carrying its own launch's tag,
 *     then clears them.  The slot is chosen on the device from the launch's
 *     grid identifier (it is not fixed when a call is captured in a CUDA
 *     graph), so launches near each other in launch order never share a slot.
 *     Two launches 32 apart in the device's launch order that run at the same
 *     time (for example on two streams, one of them issuing 32 launches while
 *     a call on the other is still running) share a slot: the writing CTA then
 *     waits in vain and reports fault bit 1 << 4 instead of adding a value from
 *     another call.  No word left by a call that faulted is ever taken by a
 *     later call.
 *   - the scratch of qmm_q4_0_smallM_noalloc (see there), 4 MiB.
 * Both stay reserved on every device that loads the library until the process
 * exits.
 *
 * Streams.  `stream` is a cudaStream_t passed as void* (NULL = legacy default
 * stream).  Work is enqueued asynchronously; a call never synchronizes.
 *
 * Overlap with the preceding kernel.  The fast-path M = 1 kernels are launched
 * as programmatic dependents of the kernel enqueued just before them on the
 * same stream: they may start, and begin streaming their WEIGHT matrices,
 * while that kernel is still finishing.  Activations are read, and outputs
 * written, only after it has completed.  Therefore the weight matrix of a call
 * must not be written by the kernel immediately preceding the call on its
 * stream; if it is, put any other stream operation in between (another
 * kernel, a memset, an event record).  Weights loaded with cudaMemcpy are
 * always safe.
 *
 * Errors.  Arguments are validated on the host before anything is launched; a
 * rejected call returns its status and launches nothing.  After a launch,
 * cudaGetLastError() != cudaSuccess returns QBW_ECUDA.  Errors raised while a
 * kernel runs surface at the caller's next synchronization, as with any CUDA
 * call.  There is no CPU fallback.
 *
 * Determinism.  Each kernel reduces in a fixed order: identical inputs give
 * bit-identical outputs from run to run.
 *
 * Fast path.  When K % 256 == 0 and the weight pointers are 16-byte aligned,
 * weight rows are streamed into shared memory with tensor copies (TMA); any
 * other K % 32 == 0 shape or alignment takes a slower, equally exact path.
 */
#ifndef QBW_H
#define QBW_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum qbw_dtype {
    QBW_F32 = 0,   /* IEEE fp32 */
    QBW_BF16 = 1   /* bfloat16 */
} qbw_dtype;

typedef enum qbw_status {
    QBW_OK = 0,
    QBW_EINVAL = 1,      /* null pointer or otherwise invalid argument */
    QBW_ESHAPE = 2,      /* M, N or K out of range, or K % 32 != 0 */
    QBW_EDTYPE = 3,      /* activation or output dtype not supported here */
    QBW_EALIGN = 4,      /* activation/output pointer not aligned to its dtype */
    QBW_ECUDA = 5,       /* a CUDA runtime call or a launch failed */
    QBW_EWORKSPACE = 6,  /* workspace missing, too small or misaligned */
    QBW_EDEVICE = 7      /* the current device is not a compute capability 10.3 GPU */
} qbw_status;

/* Human-readable name of a status code (static string, never NULL). */
const char *qbw_status_str(qbw_status s);

/* Library ABI version, (major << 16) | minor. */
uint32_t qbw_version(void);

/*
 * qmv_q8_0 -- y = W x for a Q8_0 weight matrix, one token (M == 1).
 *
 * The decode-step matrix-vector product: every weight byte is read once per
 * token (SafeC Gemma 4 design notes, "Batched decode"; jouleclaw-loader-gguf
 * BENCHMARKS, "Matmul throughput -- Q8_0 scalar vs NEON").
 *
 *   w  : N * (K/32) * 34 bytes of Q8_0 blocks, any alignment
 *   x  : K activations of dtype xt, aligned to the dtype
 *   y  : N outputs of dtype yt (QBW_F32 or QBW_BF16; bf16 is rounded to
 *        nearest-even from the fp32 accumulator)
 *   M  : must be 1                         (else QBW_ESHAPE)
 *   N  : 1 .. 2^31-1, K: 32 .. 2^24, K % 32 == 0   (else QBW_ESHAPE)
 */
qbw_status qmv_q8_0(const void *w, const void *x, qbw_dtype xt, void *y, qbw_dtype yt,
                    int64_t M, int64_t N, int64_t K, void *stream);

/*
 * qmv_q4_0 -- y = W x for a Q4_0 weight matrix, one token (M == 1).
 *
 * The bandwidth-bound decode projection (gem docs/research/architecture.md,
 * "M4 Max operating assumptions" and the "dedicated four-output-row
 * matrix-vector path" of "Ownership boundaries").  Arguments as qmv_q8_0,
 * with w holding N * (K/32) * 18 bytes of Q4_0 blocks.
 */
qbw_status qmv_q4_0(const void *w, const void *x, qbw_dtype xt, void *y, qbw_dtype yt,
                    int64_t M, int64_t N, int64_t K, void *stream);

/*
 * qmv_gateup_q4_0 -- out = gelu_tanh(Wg x) * (Wu x), one pass over both
 * matrices, one token (M == 1).
 *
 * The gated FFN's gate and up projections fused with its activation, where
 * gelu_tanh(v) = 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3))) (SafeC Gemma
 * 4 design notes, "Gated FFN"; fusing gate and up into one dispatch:
 * "Performance optimizations: fusion ..."; the GPU-chained gated GELU and its
 * large-gate regression: "Further optimization: QKV projection fusion, fully
 * GPU-chained FFN").
 *
 *   w_gate, w_up : two Q4_0 matrices of N rows and K inputs each.  A fused
 *                  [gate ; up] buffer works too: pass w_up = w_gate + N*K/32*18.
 *   x            : K activations (xt);   out : N outputs (ot)
 *   M == 1; N, K as for qmv_q4_0.
 */
qbw_status qmv_gateup_q4_0(const void *w_gate, const void *w_up, const void *x, qbw_dtype xt,
                           void *out, qbw_dtype ot, int64_t M, int64_t N, int64_t K, void *stream);

/*
 * qmm_q4_0_smallM -- Y = X W^T for a few token rows (prefill tiles), on the
 * tensor cores.
 *
 * Prompt tiles of up to 32 tokens share one read of each Q4_0 weight and run
 * on matrix units (gem docs/research/architecture.md, "Ownership
 * boundaries"); dequantize-then-matrix-unit wins from m of about 8
 * (jouleclaw-loader-gguf BENCHMARKS, "Q8_0 matmul -- NEON direct vs
 * AMX-tiled").  Weights are dequantized to bf16 on chip and multiplied in
 * bf16 with fp32 accumulation.
 *
 *   w : Q4_0 matrix, N rows x K inputs        X : [M, K] row-major, QBW_BF16
 *   Y : [M, N] row-major, QBW_BF16 or QBW_F32
 *   M : 1 .. 32 (tuned for 8, 16, 32)          N >= 1, K % 32 == 0
 *   workspace : device scratch of at least
 *               qmm_q4_0_smallM_workspace_bytes(M, N, K) bytes (size for the
 *               current device), 256-byte aligned, ZERO-FILLED once before
 *               its first use.  It holds one arrival counter per 128-row
 *               tile in a fixed 4096-byte region at its start, then either
 *               the split-K partial sums or, for M <= 16 when whole-tile
 *               splits would leave SMs idle (a stream-K plan: one CTA per SM
 *               over equal ranges of the tiles' K-groups), one tagged 64-bit
 *               word per CTA, row and token column.  Every call leaves the
 *               whole workspace zero again, so the single zero-fill at
 *               allocation is enough, also when one workspace serves calls of
 *               different shapes; after a call that reported a device fault
 *               (qbw_fault_read), zero-fill it again (a call that gave up may
 *               leave arrival counters nonzero; tagged words carry their
 *               launch's grid identifier, so no later call takes a stale
 *               one).  Calls that share one
 *               workspace must not run concurrently.  May be
 *               NULL when the size query returns 0: so it does for one K-split
 *               per tile, and for 2 .. 8 splits when the device holds all the
 *               tiles' thread-block clusters at once (the splits of a tile
 *               then add their partial sums in distributed shared memory).
 *
 * Fast path: K % 256 == 0 and w, X 16-byte aligned (tcgen05 tensor cores);
 * other shapes take an exact CUDA-core path that needs no workspace.  With
 * M <= 2 and at least 15 MB of weights the call runs on the exact-code kernel
 * of qmv_q4_0 (integer codes on the tensor cores, block scales applied in
 * fp32: no weight is rounded), which needs no workspace either.
 */
size_t qmm_q4_0_smallM_workspace_bytes(int64_t M, int64_t N, int64_t K);
qbw_status qmm_q4_0_smallM(const void *w, const void *X, qbw_dtype xt, void *Y, qbw_dtype yt,
                           int64_t M, int64_t N, int64_t K, void *workspace, size_t workspace_bytes,
                           void *stream);

/*
 * qmm_q4_0_smallM_noalloc -- qmm_q4_0_smallM without a workspace argument, for
 * callers that cannot allocate device memory at the call (an engine that has
 * handed all of HBM to weights and KV cache up front, a plain C host program
 * with no device allocator of its own).  The published descriptions of the
 * method have no counterpart to this call; it is a convenience of this library.
 *
 * The split-K scratch is a static device array of QBW_QMM_NOALLOC_SCRATCH_BYTES
 * inside the library; nothing is allocated or freed.  A request that needs more
 * scratch than that (qmm_q4_0_smallM_workspace_bytes(M, N, K) > the limit)
 * returns QBW_EWORKSPACE and launches nothing.  On a 152-SM GB300 every legal
 * shape needs at most 2,494,464 bytes, so the limit is only reached on parts
 * with more SMs.
 *
 * Every call that needs scratch looks up the array's address on the current
 * device (cudaGetSymbolAddress; no allocation).  The first such call on a
 * device, and the first one after qbw_fault_read has reported a nonzero fault
 * word, first zero-fills the array on `stream` (cudaMemsetAsync): the arrival
 * counters must start at zero, every completed call leaves them at zero, but a
 * call that gave up on a bounded wait may leave them nonzero.  Make the first
 * call before any stream capture, and read the fault word outside a capture.
 *
 * All calls on one device share the one array: calls that may overlap in time
 * (different streams without ordering, several host threads) race on it and
 * give wrong results.  Arguments, results and errors are otherwise those of
 * qmm_q4_0_smallM, and the results are bit-identical to it.
 */
#define QBW_QMM_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20)
qbw_status qmm_q4_0_smallM_noalloc(const void *w, const void *X, qbw_dtype xt, void *Y, qbw_dtype yt,
                                   int64_t M, int64_t N, int64_t K, void *stream);

/*
 * qdequant_q8_0 / qdequant_q4_0 -- expand a whole matrix to fp32:
 * out[n*K + k] = w[n, k].  Every product d*q is exact in fp32, so the result is
 * bit-exact.  Meant for testing and inspection, not for the hot path.
 *
 *   w : N rows of K/32 blocks, any alignment;   out : N*K floats, 4-byte aligned
 */
qbw_status qdequant_q8_0(const void *w, float *out, int64_t N, int64_t K, void *stream);
qbw_status qdequant_q4_0(const void *w, float *out, int64_t N, int64_t K, void *stream);

/*
 * qmv_q4_k -- y = W x for a Q4_K weight matrix, one token (M == 1).
 *
 * Q4_K, the K-quant the pages benchmark beside Q8_0 (jouleclaw-loader-gguf
 * BENCHMARKS, "Q4_K matmul -- scalar fused vs AMX-tiled" and its NEON
 * follow-up): super-blocks of 256 weights in 144 bytes, the GGUF block_q4_K
 * record -- fp16 d, fp16 dmin, 12 bytes of six-bit sub-block scales sc_j and
 * mins m_j (j = 0..7, 32 weights each), 128 bytes of 4-bit codes q (each
 * 64-weight chunk keeps its first 32 codes in the low nibbles of its 32
 * bytes and the rest in the high nibbles).  w = d sc_j q - dmin m_j.  Each
 * sub-block is summed by the pages' algebraic split,
 * d sc_j * sum(q x) - dmin m_j * sum(x).
 *
 *   w : N rows of K/256 super-blocks (row stride K/256 * 144 bytes)
 *   x, y, xt, yt, M, N as for qmv_q4_0;  K % 256 == 0 (else QBW_ESHAPE)
 *
 * Fast path: w and x 16-byte aligned (tcgen05 tensor cores, exact integer
 * codes); otherwise an exact CUDA-core kernel.
 */
qbw_status qmv_q4_k(const void *w, const void *x, qbw_dtype xt, void *y, qbw_dtype yt,
                    int64_t M, int64_t N, int64_t K, void *stream);

/*
 * qdequant_q4_k -- expand a Q4_K matrix to fp32: out[n*K + k] = w[n, k], the
 * nearest fp32 to the exact d sc_j q - dmin m_j (d sc_j q and dmin m_j are
 * exact in fp32; their difference is rounded once).  For testing.
 *
 *   w : N rows of K/256 super-blocks, any alignment;  out : N*K floats, 4-byte
 *   aligned;  K % 256 == 0 (else QBW_ESHAPE)
 */
qbw_status qdequant_q4_k(const void *w, float *out, int64_t N, int64_t K, void *stream);

/*
 * Mixed-bit matrices -- int2-symmetric, int4-affine and int8 weights as a QAT
 * checkpoint ships them for hand-written decode kernels (Core AI model zoo,
 * Gemma-4-E2B raw-Metal port, "What shipped" and "Architecture": mixed-bit
 * matvecs over quantized words qp, scales sc and biases bi).  The page gives
 * no byte layout; this library reads the following one.
 *
 *   qp : N rows of K * b / 32 little-endian 32-bit words, rows back to back;
 *        weight k of a row is bits [(k b) % 32, (k b) % 32 + b) of word
 *        (k b) / 32 of that row (b = 2, 4, 8; lowest bits first)
 *   sc : fp16 scales, one per group of `group` consecutive weights of a row,
 *        [N][K / group] row-major
 *   bi : fp16 biases, same shape as sc (int4-affine only; ignored otherwise)
 *   QBW_MIXBIT_INT2_SYM    : q = the field as a two's-complement 2-bit value
 *                            (-2 .. 1), w = sc q
 *   QBW_MIXBIT_INT4_AFFINE : c = the field as unsigned (0 .. 15), w = sc c + bi
 *   QBW_MIXBIT_INT8_SYM    : q = the field as a two's-complement byte, w = sc q
 *
 * Ranges: group a multiple of 16 dividing K; K * b a multiple of 128 (rows of
 * whole 16-byte word groups: K % 64 for 2 bits, % 32 for 4, % 16 for 8), else
 * QBW_ESHAPE.  qp 16-byte aligned, sc and bi 4-byte aligned (QBW_EALIGN).
 */
typedef enum qbw_mixbit {
    QBW_MIXBIT_INT2_SYM = 2,
    QBW_MIXBIT_INT4_AFFINE = 4,
    QBW_MIXBIT_INT8_SYM = 8
} qbw_mixbit;

/*
 * qmv_mixbit -- y = W x for a mixed-bit matrix, one token (M == 1).  The int4
 * form is summed as sc * sum(c x) + bi * sum(x) per group, so its rounding
 * scales with sum (|sc c| + |bi|) |x|.
 *
 * Groups of 32 (or a larger power of two), K % 256 == 0, sc (and bi) 16-byte
 * aligned and at least 5 MB (int4), 4 MB (int2) or 16 MB (int8) of codes (10,
 * 5 and 64 MB when K <= 4096) run on the tensor cores where their launch plan
 * takes the shape (its row tiles and K-groups per CTA are bounded;
 * qmv_mixbit_route reports the outcome), like qmv_q4_k: the
 * codes enter the MMA exactly (int8 as its low nibble and its signed high
 * nibble), x as two (bf16) or three (fp32) e4m3 pieces per element under a
 * power-of-two scale per 32 elements, and the rows whose pieces may miss more
 * than 2^-11 of sum |sc q x| get the missed part added exactly; they use the
 * split-tile scratch above.  Every other call takes the CUDA-core kernel.
 *
 *   x : K activations of xt, 16-byte aligned;  y : N outputs of yt
 *   M == 1; N >= 1; K as above.  On the CUDA-core kernel K must also be small
 *   enough that the activations (4 K bytes, 4.5 K for int4) and the copy rings
 *   (40 to 98 KB; the larger rings only for K <= 8192) fit one CTA's shared
 *   memory (227 KB): K up to 37,000 in every format and group size, else
 *   QBW_ESHAPE.  Calls that take the tensor cores have no such bound.
 */
qbw_status qmv_mixbit(qbw_mixbit kind, const void *qp, const void *sc, const void *bi, int64_t group,
                      const void *x, qbw_dtype xt, void *y, qbw_dtype yt, int64_t M, int64_t N, int64_t K,
                      void *stream);

/*
 * qmv_mixbit_route -- which kernel qmv_mixbit takes for these arguments on the
 * current device: *tensor_cores = 1 for the tensor-core form, 0 for the
 * CUDA-core kernel.  For testing.  Arguments as qmv_mixbit (xt the activation
 * type); returns the status qmv_mixbit's argument checks would give, before
 * any launch.  Launches nothing.
 */
qbw_status qmv_mixbit_route(qbw_mixbit kind, const void *qp, const void *sc, const void *bi, int64_t group,
                            qbw_dtype xt, int64_t N, int64_t K, int *tensor_cores);

/*
 * qdequant_mixbit -- out[n*K + k] = w[n, k] in fp32 (sc q exactly; sc c + bi
 * rounded once to nearest).  For testing.  Arguments as qmv_mixbit; out 4-byte
 * aligned.
 */
qbw_status qdequant_mixbit(qbw_mixbit kind, const void *qp, const void *sc, const void *bi, int64_t group,
                           float *out, int64_t N, int64_t K, void *stream);

/*
 * qembed_q8_0 -- token-table lookup: out[i, :] = W[ids[i], :], dequantized.
 *
 * The embedding side of the Q8_0 token table that the decode loop reads once
 * per token (gem docs/research/architecture.md, "M4 Max operating
 * assumptions": Q4_0 matrices and a Q8_0 token table; the same table serves
 * as the tied LM head through qmv_q8_0).
 *
 *   w   : Q8_0 matrix, N rows x K inputs, any alignment
 *   ids : n_ids row indices (int32, device memory, 4-byte aligned)
 *   out : [n_ids, K] of ot; QBW_F32 holds d * q exactly, QBW_BF16 that value
 *         rounded to nearest even
 *   n_ids >= 0 (0 launches nothing; ids and out may then be NULL), N >= 1,
 *   K % 32 == 0
 * An index outside [0, N) gives a row of zeros and sets fault bit 1 << 3
 * (see qbw_fault_read); nothing is read out of bounds.
 */
qbw_status qembed_q8_0(const void *w, const int32_t *ids, int64_t n_ids, void *out, qbw_dtype ot, int64_t N,
                       int64_t K, void *stream);

/*
 * Chained products -- a sequence of dependent Q4_0 matrix-vector products in
 * one launch, such as one token's decode weight sweep (per layer q|k|v, o,
 * gate+up, down, each step's activations the previous step's output).  The
 * pages count the GPU round trips per token and chain the FFN's dispatches
 * on the GPU to cut them, against one command buffer per token as the
 * reference point (SafeC Gemma 4 design notes, "Further optimization: QKV
 * projection fusion, fully GPU-chained FFN").
 *
 * Defined by the same arithmetic as qmv_q4_0 / qmv_gateup_q4_0 with M = 1 and
 * bf16 activations: step s computes y_s = W_s x_s, or, when w_up is given,
 * y_s = gelu_tanh(W_s x_s) * (W_up,s x_s), with the weights of the Q4_0
 * layout above.  Steps run in order and step s sees
 * the outputs of every earlier step, so x_s may be (part of) an earlier y.
 * The results match the separate calls within the same bound (2e-3 of the
 * row's sum |w x|, plus the bf16 output rounding).
 *
 * qbw_chain_step (one step; the caller keeps every buffer alive and in place
 * while the chain exists):
 *   w    : Q4_0 matrix, N rows of K/32 blocks, 16-byte aligned (QBW_EALIGN)
 *   w_up : NULL for y = W x; else the up matrix, same shape and alignment
 *   x    : bf16 [K], 16-byte aligned; may not overlap this step's y (QBW_EINVAL)
 *   y    : [N] of yt (QBW_BF16 or QBW_F32, else QBW_EDTYPE), aligned to yt;
 *          may not overlap any step's weights (QBW_EINVAL)
 *   N    : 1 .. 2^31-1;  K: 256 .. 2^24, K % 256 == 0 (else QBW_ESHAPE); a
 *          step whose unit split exceeds the kernel's per-CTA capacity (far
 *          beyond the model shapes) also gives QBW_ESHAPE
 *
 * qbw_chain_create -- validate nsteps >= 1 steps (QBW_EINVAL for a null or
 *   empty list), encode their weight descriptors and copy them, with a
 *   barrier counter and split-tile scratch, to memory it allocates on the
 *   current device (QBW_ECUDA if that fails).  *out receives the chain,
 *   owned by the caller until qbw_chain_destroy.
 * qbw_chain_run -- enqueue the whole chain on `stream` (a CUDA stream of the
 *   chain's device, else QBW_EINVAL): a counter reset and one cooperative
 *   launch with one CTA per SM, so it may be captured in a CUDA graph.  Runs
 *   of one chain must not overlap in time (they share its counter and
 *   scratch).  Device-side problems set fault-word bits (see qbw_fault_read).
 * qbw_chain_destroy -- free the chain's device memory (after its last run has
 *   completed) and the chain.
 */
typedef struct qbw_chain_step {
    const void *w;
    const void *w_up;
    const void *x;
    void *y;
    qbw_dtype yt;
    int64_t N;
    int64_t K;
} qbw_chain_step;

typedef struct qbw_chain_s *qbw_chain;

qbw_status qbw_chain_create(const qbw_chain_step *steps, int nsteps, qbw_chain *out);
qbw_status qbw_chain_run(qbw_chain chain, void *stream);

/*
 * qbw_chain_run_launches -- enqueue the chain as one kernel launch per step
 * on `stream` (the tensor-core kernel of qmv_q4_0 / qmv_gateup_q4_0, each
 * launched as a programmatic dependent of the one before), instead of one
 * cooperative launch.  Each step's results are bit-identical to the separate
 * call; what the chain adds is that every launch, once it has issued its last
 * weight copy, prefetches into L2 the first weight tiles its CTAs will load in
 * the next step, so the next launch's first copies come from L2 rather than
 * HBM.  May be captured in a CUDA graph.  QBW_EINVAL as for qbw_chain_run;
 * QBW_ESHAPE for a step the tensor-core kernel does not take (more than
 * 524,288 rows).  Allocates nothing; the chain's own scratch is not used.
 */
qbw_status qbw_chain_run_launches(qbw_chain chain, void *stream);
qbw_status qbw_chain_destroy(qbw_chain chain);

/*
 * qbw_fault_read -- read the library's device fault word for the current
 * device.  Kernels report problems found while they run by setting bit
 * (1 << c) of this word, then return early (outputs of that call are then
 * undefined) instead of hanging or trapping:
 *   c = 1  a bounded wait for an asynchronous copy ran out (about two seconds)
 *   c = 2  a bounded wait for tensor-core work ran out
 *   c = 3  qembed_q8_0 met a row index outside [0, N)
 *   c = 4  a kernel waited in vain (about two seconds) for another CTA's share
 *          of a 128-row tile split between CTAs (qmv_q4_0, qmv_gateup_q4_0,
 *          qmv_q4_k, qmm_q4_0_smallM; see "Library state" for the one case
 *          of concurrent launches that causes it)
 *   c = 5  internal: a launch plan exceeded a kernel's fixed capacity (the
 *          host-side planning never allows it; seen only after a library bug)
 *   c = 6  qbw_chain_run: a CTA waited in vain (about two seconds) for the
 *          other CTAs at the barrier between two steps
 * Synchronizes `stream`, stores the word in *code and, if clear != 0, resets
 * it to zero.
 */
qbw_status qbw_fault_read(uint32_t *code, int clear, void *stream);

/*
 * qbw_selftest_wait -- test-only: run one of the library's bounded waits on
 * something nothing completes, with a limit of limit_us microseconds (1 ..
 * 2,000,000), so a test can check that the wait gives up, that its code
 * reaches the fault word and that the device stays usable.  The pages have no
 * counterpart; it exercises this library's failure detection.
 *   which = 0: phase 0 of a fresh shared-memory mbarrier (the wait of every
 *              copy and MMA stage): sets fault bit 1 << 1
 *   which = 1: the tag of a global word that stays 0 (the split-tile share
 *              wait of qmv_q4_0 / qmv_q4_k): sets fault bit 1 << 4
 * Enqueues one tiny kernel on `stream` and returns; QBW_EINVAL for other
 * arguments.
 */
qbw_status qbw_selftest_wait(int which, uint32_t limit_us, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* QBW_H */
