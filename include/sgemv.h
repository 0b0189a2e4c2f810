/*
 * sgemv.h -- C ABI of the GB300 INT4 + 2:4 "2bit-CSR" SparseGemv library (libsgemv.so).
 *
 * The library computes the decode-time product y = W x of the paper "Efficient LLM-based Advertising
 * via Model Compression and Parallel Verification" (§3.3 "Revised Kernel"), where W is stored with
 *   - group-wise INT4 weight-only quantisation, fp16 scale and integer zero point per group, one group
 *     size per layer (§1 "Our Main Idea"; §3.2 "Adaptive Group-Wise Quantization"), and
 *   - for sparse layers, 2:4 semi-structured sparsity encoded as "2bit-CSR": the kept values plus a
 *     2-bit in-block position per kept value, packed least-significant-first into uint16_t words
 *     (§1 Contributions; §3.2 "Sparsification"; §3.3 "Sparse Index Structure" and "Reduce
 *     Computational Burden").
 * Layers that the layer-adaptive policy leaves dense use the dense INT4 variant, the "previous
 * generation Gemv" the paper's SparseGemv refines (§3.3 opening paragraph).
 * The byte layout of a packed layer is the packed format, version 1 (sections cited below).
 *
 * Conventions for every function below:
 *   - Return value: SGEMV_OK (0) or a negative SGEMV_ERR_* code. Functions never throw, never
 *     allocate or free memory, and never synchronise a stream or the device.
 *   - Argument errors are detected on the host before anything is launched; nothing is launched
 *     when an error is returned.
 *   - Device pointers ("_dev") are CUDA global-memory addresses on the current device, owned by the
 *     caller, and must be 16-byte aligned (a packed buffer: 32-byte aligned). The library keeps no
 *     reference to them after the call.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream). Work is
 *     enqueued on it asynchronously; the caller keeps every buffer alive until that work completes.
 *   - `status_dev` (nullable) is a device int32 that device code sets to a negative SGEMV_ERR_* code
 *     if it detects an error while running (non-finite weights at pack time, bad beam inputs). It is
 *     never reset by the library: initialise it to 0 and read it after the stream has completed.
 *   - The library is stateless apart from a per-device cache of kernel attributes; it is safe to call
 *     from several host threads.
 */
#ifndef SGEMV_H
#define SGEMV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
enum {
    SGEMV_OK = 0,
    SGEMV_ERR_ARG = -1,       /* null pointer, bad batch, bad enum value, short buffer */
    SGEMV_ERR_SHAPE = -2,     /* N, K or group size outside the limits of packed format v1, section 1
                                 (for sparse formats also N * kept elements per row > 2^31 - 1) */
    SGEMV_ERR_ALIGN = -3,     /* a pointer is not 16-byte (packed buffer: 32-byte) aligned */
    SGEMV_ERR_FORMAT = -4,    /* layout/header mismatch, or a sparse layer given to the dense call */
    SGEMV_ERR_CUDA = -5,      /* a CUDA runtime call (launch, attribute query) failed */
    SGEMV_ERR_NONFINITE = -6, /* device-reported: the weights contain inf or NaN */
    SGEMV_ERR_TIMEOUT = -7    /* device-reported by sgemv_run_stack: a bounded wait for the copy engine's
                                 copy of x gave up (the launch's y is then invalid) */
};

/* Packed formats (packed format v1, section 2). */
enum {
    SGEMV_FMT_SPARSE24 = 1, /* 2:4 sparse INT4 in 2bit-CSR, read by sgemv_run */
    SGEMV_FMT_DENSE = 2,    /* dense INT4, read by sgemv_run_dense */
    SGEMV_FMT_SPARSE14 = 3  /* 1:4 sparse INT4 in 2bit-CSR (Table 1 "Sparse(1:4)"), read by sgemv_run */
};

/*
 * Where each section of a packed layer lives (packed format v1, sections 3-4). All offsets are in bytes from
 * the start of the packed buffer; pitches are bytes per weight row of that section.
 */
typedef struct {
    int32_t format, n, k, group;
    uint64_t vals_pitch, idx_pitch, sz_pitch;
    uint64_t off_vals, off_idx, off_sz, off_rowptr, total_bytes;
} sgemv_layout;

/*
 * sgemv_layout_query -- host only, pure. Fills *out with the layout of an N x K layer of the given
 * format and group size. Errors: SGEMV_ERR_ARG (out is NULL or format unknown), SGEMV_ERR_SHAPE.
 * The caller allocates `out->total_bytes` bytes of device memory for the packed layer.
 */
int sgemv_layout_query(int format, int n, int k, int group, sgemv_layout* out);

/*
 * sgemv_pack -- compress an fp16 weight matrix on the GPU (the offline step of §3.2-§3.3: 2:4 or 1:4
 * magnitude pruning for SPARSE24 / SPARSE14, group-wise INT4 quantisation, 2bit-CSR encoding).
 *   layout     : from sgemv_layout_query (its format selects sparse or dense packing).
 *   w_dev      : fp16 W[n][k], row-major, read only.
 *   packed_dev : output, layout->total_bytes bytes; every byte is written (padding is zero), so the
 *                result is bit-identical from run to run and to the CPU oracle's packing.
 *   status_dev : nullable; set to SGEMV_ERR_NONFINITE if W holds inf or NaN (the packed bytes are then
 *                unspecified).
 * Errors returned: SGEMV_ERR_ARG, SGEMV_ERR_FORMAT (layout fields inconsistent), SGEMV_ERR_ALIGN,
 * SGEMV_ERR_CUDA.
 */
int sgemv_pack(const sgemv_layout* layout, const void* w_dev, void* packed_dev, int32_t* status_dev,
               void* stream);

/*
 * sgemv_run -- the SparseGemv of §3.3: y[b][i] = sum_j Ŵ[i][j] * x[b][j] for a SPARSE24 or SPARSE14
 * layer, with Ŵ = (q - z) * s at the kept positions (packed format v1, section 6), accumulated in fp32.
 *   layout     : layout of the packed layer (SGEMV_FMT_SPARSE24 or SGEMV_FMT_SPARSE14).
 *   packed_dev : the packed layer written by sgemv_pack (read only).
 *   x_dev      : fp16 x[batch][k], row-major (read only). batch is the beam width, 1..8.
 *   y_dev      : fp16 y[batch][n], row-major, written (round to nearest even from fp32). y may overlap
 *                neither x nor the packed buffer (SGEMV_ERR_ARG).
 *   status_dev : nullable, 4-byte aligned. The GEMV detects no errors on the device and never writes it.
 * The kernel uses programmatic dependent launch: it may ask L2 to prefetch its weights while the
 * previous kernel on `stream` is still running, and reads x and the weights only after that kernel
 * has completed.
 * Reproducibility: a layer that streams -- batch 1..3, not split over K, and its x (all batch rows)
 * fits a CTA's shared memory -- sums each row in a fixed order, so its y is bit-identical from run to
 * run. Batch 4..8, a layer split over K (fewer rows than half the SMs and K >= 32768) or one whose x
 * does not fit runs the tiled kernel, whose warps add their row sums with shared-memory atomics: its y
 * may differ from run to run in the last bits (always within the accuracy bound).
 * Errors returned: SGEMV_ERR_ARG, SGEMV_ERR_FORMAT (not a sparse layout, or inconsistent fields),
 * SGEMV_ERR_ALIGN, SGEMV_ERR_CUDA.
 */
int sgemv_run(const sgemv_layout* layout, const void* packed_dev, const void* x_dev, int batch,
              void* y_dev, int32_t* status_dev, void* stream);

/*
 * sgemv_run_dense -- the dense INT4 weight-only GEMV ("previous generation Gemv", §3.3) for a DENSE
 * layer. Arguments, semantics and errors as sgemv_run; the layout must be SGEMV_FMT_DENSE.
 */
int sgemv_run_dense(const sgemv_layout* layout, const void* packed_dev, const void* x_dev, int batch,
                    void* y_dev, int32_t* status_dev, void* stream);

/*
 * One row of the per-layer dispatch table (the layer-adaptive policy of §3.1-§3.2: each layer has
 * its own format and group size). x_dev/y_dev are that layer's input and output; a caller that chains
 * layers points a layer's x_dev at the previous layer's y_dev.
 */
typedef struct {
    sgemv_layout layout;
    const void* packed_dev;
    const void* x_dev;
    void* y_dev;
} sgemv_layer;

/*
 * sgemv_run_stack -- run every layer of the table in order on `stream`, each with the kernel its
 * format selects (sgemv_run or sgemv_run_dense), all with the same batch. Consecutive layers of the same
 * format with no data flow between them (no layer's x overlaps an earlier member's y, no y overlaps an
 * earlier member's x or y) run as one launch of up to 8 layers: each CTA works through its rows of all of
 * them as one list, so the launch gap, the dependent-launch wait and the tail are paid once per group.
 * The table is read on the host during the call only. Validation covers every row before the first
 * launch; on an error no layer is launched. Errors: as sgemv_run; SGEMV_ERR_ARG also for a NULL table
 * or n_layers < 1.
 * status_dev: nullable, 4-byte aligned. A launch of several layers fetches their x with the copy engine
 * (one bulk copy per layer and batch row) and waits for it with a bounded wait; if that wait gives up,
 * SGEMV_ERR_TIMEOUT is stored here. Nothing else is written.
 */
int sgemv_run_stack(const sgemv_layer* table, int n_layers, int batch, int32_t* status_dev,
                    void* stream);

/*
 * sgemv_header_read -- host only. Parses the 64-byte header at the start of a packed buffer (a host
 * copy of at least 64 bytes) and fills *out. Use it when loading a persisted packed layer.
 * Errors: SGEMV_ERR_ARG (NULL or bytes < 64), SGEMV_ERR_FORMAT (bad magic, version or offsets),
 * SGEMV_ERR_SHAPE.
 */
int sgemv_header_read(const void* header_host, uint64_t bytes, sgemv_layout* out);

/*
 * sgemv_header_check -- host only. SGEMV_OK if the header copy describes exactly `layout`,
 * SGEMV_ERR_FORMAT otherwise (SGEMV_ERR_ARG for NULL or bytes < 64).
 */
int sgemv_header_check(const sgemv_layout* layout, const void* header_host, uint64_t bytes);

/*
 * The prefix tree of the tree-based parallel verification (§3.4 "Tree-Based Parallel Verification"),
 * in CSR form on the device. Node 0 is the root. The children of node u are the edges
 * child_ptr[u] .. child_ptr[u+1]-1; edge e carries token child_tok[e] and leads to node child_node[e].
 * The edges of a node are stored in ascending token order. All arrays are int32, owned by the caller.
 */
typedef struct {
    int32_t n_nodes;               /* >= 1; child_ptr has n_nodes + 1 entries */
    int32_t n_edges;               /* child_tok and child_node have n_edges entries */
    const int32_t* child_ptr_dev;
    const int32_t* child_tok_dev;
    const int32_t* child_node_dev;
} sgemv_trie;

/*
 * sgemv_beam_step -- one trie-constrained beam-score step (§3.4): the decoder's scores are filtered by
 * the trie to the children of each beam's node, each child's score is B = score[b] + logp[b][token]
 * (one binary32 addition: logp holds log-probabilities, so the paper's "logarithmic summation" is a
 * sum), and the best `k` candidates are kept.
 *   trie          : the prefix tree (device arrays).
 *   beam_in       : input beams, 1..64. node_dev[b] (int32) is beam b's trie node, score_dev[b] (fp32)
 *                   its score.
 *   vocab, logp_dev : fp32 logp[beam_in][vocab], row-major (the decoder's log-probabilities for each
 *                   input beam's next position).
 *   k             : beams to keep, 1..64.
 *   out_*_dev     : the kept candidates in rank order (each array k entries; entries from *out_count_dev
 *                   on are unspecified): trie node (int32), score (fp32), input beam (int32), token
 *                   (int32); *out_count_dev = min(k, valid candidates).
 *   status_dev    : nullable; SGEMV_ERR_NONFINITE if a NaN score was dropped, SGEMV_ERR_ARG if a node id
 *                   or token is out of range (those candidates are dropped), SGEMV_ERR_SHAPE if the step
 *                   has more than 16384 candidates (nothing is kept: *out_count_dev = 0).
 * Ranking: score descending; ties go to the lower input beam, then the lower token. -inf scores
 * (probability 0) are candidates and rank last. One CTA, asynchronous on `stream`.
 * Errors returned: SGEMV_ERR_ARG (NULL pointers, counts out of range), SGEMV_ERR_ALIGN (a pointer not
 * 4-byte aligned), SGEMV_ERR_CUDA.
 */
int sgemv_beam_step(const sgemv_trie* trie, int beam_in, int vocab, const int32_t* node_dev,
                    const float* score_dev, const float* logp_dev, int k, int32_t* out_node_dev,
                    float* out_score_dev, int32_t* out_parent_dev, int32_t* out_tok_dev, int32_t* out_count_dev,
                    int32_t* status_dev, void* stream);

/*
 * sgemv_beam_traceback -- the final traceback of §3.4: seq[f][t] (int32, [beam_max][steps]) is the
 * token of final beam f at step t, following parent links back from the last step.
 *   parent_dev, tok_dev : int32 [steps][beam_max]: row t holds the out_parent / out_tok of step t.
 *   count_dev           : int32, the last step's out_count; rows f >= count are filled with -1.
 *   status_dev          : nullable; SGEMV_ERR_ARG if a parent link is out of range (that row gets -1).
 * beam_max is 1..64. Errors returned: SGEMV_ERR_ARG, SGEMV_ERR_ALIGN, SGEMV_ERR_CUDA.
 */
int sgemv_beam_traceback(int steps, int beam_max, const int32_t* parent_dev, const int32_t* tok_dev,
                         const int32_t* count_dev, int32_t* seq_dev, int32_t* status_dev, void* stream);

/*
 * sgemv_beam_decode -- a whole decode of the tree-based verification (§3.4) in one launch: `steps`
 * beam-score steps (each exactly as sgemv_beam_step) and the traceback. It applies when the decoder's
 * distributions for every position are known before the beam search, as in the paper's parallel
 * verification, where one forward pass scores all positions.
 *   beam_in, node_dev, score_dev : the input beams of step 0 (as in sgemv_beam_step).
 *   logp_dev      : HOST array of `steps` device pointers (1..32 steps). Step t reads its input beam b's
 *                   log-probabilities at logp_dev[t] + b * logp_stride; logp_stride is vocab (one row per
 *                   input beam: room for k rows, beam_in rows at step 0) or 0 (one row, the position's
 *                   distribution, shared by all beams).
 *   k             : beams kept per step, 1..64. Step t's input beams are step t-1's kept beams.
 *   out_*_dev     : per-step outputs as in sgemv_beam_step, [steps][k] (row t = step t); out_count_dev
 *                   [steps].
 *   seq_dev       : int32 [k][steps]: the traceback of the final beams (as sgemv_beam_traceback; rows
 *                   from the final count on are -1).
 *   status_dev    : nullable; as in sgemv_beam_step, for any step.
 * The ranking and every output are bit-identical to the steps run one by one through sgemv_beam_step and
 * sgemv_beam_traceback. One CTA, asynchronous on `stream`.
 * Errors returned: SGEMV_ERR_ARG (NULL pointers, counts out of range, logp_stride not 0 or vocab),
 * SGEMV_ERR_ALIGN (a pointer not 4-byte aligned), SGEMV_ERR_CUDA.
 */
int sgemv_beam_decode(const sgemv_trie* trie, int steps, int vocab, int beam_in, const int32_t* node_dev,
                      const float* score_dev, const float* const* logp_dev, int logp_stride, int k,
                      int32_t* out_node_dev, float* out_score_dev, int32_t* out_parent_dev, int32_t* out_tok_dev,
                      int32_t* out_count_dev, int32_t* seq_dev, int32_t* status_dev, void* stream);

/* Human-readable name of a status code (static string, never NULL). */
const char* sgemv_status_str(int status);

/* Library ABI version (1). */
int sgemv_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SGEMV_H */
