// Trie-constrained beam-score step and traceback: the decoding side of the tree-based parallel
// verification of the paper "Efficient LLM-based Advertising via Model Compression and Parallel
// Verification" (§3.4 "Tree-Based Parallel Verification"): the decoder's per-position scores are
// filtered by the prefix tree to the valid next tokens, each valid token's log-probability is added to
// its parent's score (B_score), beam search keeps the best `k` nodes, and at the last position the
// kept nodes are traced back into token sequences.
//
// One CTA of 1024 threads per step (the candidate set is small: beam_in x children). Candidates are
// numbered in (input beam, edge) order; each gets the 64-bit key (rank of its score, descending) << 32 |
// its number, so one ascending bitonic sort (shared memory plus warp shuffles) ranks them by score and
// breaks ties by the lower input beam, then the lower token (edges of a node are in ascending token
// order). Scores are
// single binary32 additions, so the ranking is bit-for-bit reproducible. Both kernels use programmatic
// dependent launch (they read nothing before griddepcontrol.wait). No waits other than __syncthreads.
#include <atomic>
#include <cstdint>
#include <cstring>

#include "common.cuh"

namespace sgemv {

namespace {

constexpr int kBeamThreads = 1024;

struct BeamParams {
    const int32_t* child_ptr;
    const int32_t* child_tok;
    const int32_t* child_node;
    int32_t n_nodes, n_edges;
    int32_t beam_in, vocab, k;
    const int32_t* node;
    const float* score;
    const float* logp;      // row b (input beam b) at logp + b * logp_stride
    int32_t logp_stride;    // vocab (one row per input beam) or 0 (one row shared by all beams)
    int32_t* out_node;
    float* out_score;
    int32_t* out_parent;
    int32_t* out_tok;
    int32_t* out_count;
    int32_t* status;
    int32_t max_cand;       // capacity of the key array (a power of two)
};

// Monotone map of binary32 to uint32 (larger float -> larger integer); -0 is treated as +0.
__device__ __forceinline__ uint32_t orderable(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7FFFFFFFu) == 0) u = 0;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ void set_status(int32_t* status, int code) {
    if (status != nullptr) atomicCAS(status, 0, code);
}

// Input beam of candidate i: the last b with off[b] <= i (off is an exclusive prefix sum).
__device__ __forceinline__ int beam_of(const int32_t* off, int beam_in, int i) {
    int lo = 0, hi = beam_in - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (off[mid] <= i) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// The bitonic steps of partner distance j < 32 of the lengths len_lo..len_hi (powers of two), for every
// key of keys[0, size) (size a multiple of 32): each thread holds key i = tid + m * kBeamThreads, whose
// partner i ^ j is held by lane (tid ^ j) of the same warp. Ends with a CTA barrier.
__device__ __forceinline__ void warp_bitonic(uint64_t* keys, int size, int tid, int len_lo, int len_hi) {
    for (int i = tid; i < size; i += kBeamThreads) {  // whole warps take part (size % 32 == 0)
        uint64_t v = keys[i];
        for (int len = len_lo; len <= len_hi; len <<= 1) {
            const bool up = (i & len) == 0;
            for (int j = (len >> 1) < 16 ? (len >> 1) : 16; j > 0; j >>= 1) {
                const uint64_t w = __shfl_xor_sync(0xFFFFFFFFu, v, j);
                const bool keep_min = ((i & j) == 0) == up;  // the lower index of an ascending pair
                v = keep_min ? (v < w ? v : w) : (v < w ? w : v);
            }
        }
        keys[i] = v;
    }
    __syncthreads();
}

// Shared-memory working set of one step.
struct StepSmem {
    uint64_t* keys;        // [max_cand]
    float* cand_score;     // [max_cand]
    int32_t* off;          // [kMaxBeam + 1]
    int32_t* first;        // [kMaxBeam]
    int32_t* n_nan;
    // optional copies of the step's output beams in shared memory (nullptr: global outputs only)
    int32_t* beam_node;    // [kMaxBeam]
    float* beam_score;     // [kMaxBeam]
    int32_t* beam_parent;  // [kMaxBeam]
    int32_t* beam_tok;     // [kMaxBeam]
};

// One beam-score step by the whole CTA; returns the number of output beams (the same in every thread).
// Ends after the output writes, without a barrier.
__device__ int beam_step_body(const BeamParams& p, const StepSmem& sm) {
    uint64_t* keys = sm.keys;
    float* cand_score = sm.cand_score;
    int32_t* off = sm.off;
    int32_t* first = sm.first;
    int32_t& n_nan = *sm.n_nan;
    const int tid = threadIdx.x;

    if (tid == 0) n_nan = 0;
    // children of every input beam's node (an invalid node id has none and is reported)
    if (tid < p.beam_in) {
        const int u = p.node[tid];
        int cnt = 0, e0 = 0;
        if (u >= 0 && u < p.n_nodes) {
            e0 = p.child_ptr[u];
            cnt = p.child_ptr[u + 1] - e0;
            if (e0 < 0 || cnt < 0 || e0 + cnt > p.n_edges) {
                cnt = 0;
                set_status(p.status, SGEMV_ERR_ARG);
            }
        } else {
            set_status(p.status, SGEMV_ERR_ARG);
        }
        first[tid] = e0;
        off[tid + 1] = cnt;
    }
    __syncthreads();
    if (tid < 32) {  // off[b + 1] = children of beams 0..b: a warp scan, two beams per lane (beam_in <= 64)
        const int c0 = 2 * tid < p.beam_in ? off[2 * tid + 1] : 0;
        const int c1 = 2 * tid + 1 < p.beam_in ? off[2 * tid + 2] : 0;
        int incl = c0 + c1;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int t = __shfl_up_sync(0xFFFFFFFFu, incl, d);
            if (tid >= d) incl += t;
        }
        const int base = incl - c0 - c1;
        if (2 * tid < p.beam_in) off[2 * tid + 1] = base + c0;
        if (2 * tid + 1 < p.beam_in) off[2 * tid + 2] = base + c0 + c1;
        if (tid == 0) off[0] = 0;
    }
    __syncthreads();
    const int n = off[p.beam_in];
    if (n > p.max_cand) {  // more candidates than the key array holds: report, emit nothing
        if (tid == 0) {
            set_status(p.status, SGEMV_ERR_SHAPE);
            *p.out_count = 0;
        }
        return 0;
    }
    int size = 32;  // a whole number of warps (the key array holds kMaxCandidates >= 32 keys)
    while (size < n) size <<= 1;

    // keys: (~rank(score) << 32) | candidate number; NaN scores and padding sort last
    for (int i = tid; i < size; i += kBeamThreads) {
        uint64_t key = ~0ull;
        if (i < n) {
            const int b = beam_of(off, p.beam_in, i);
            const int e = first[b] + (i - off[b]);
            const int tok = p.child_tok[e];
            if (tok >= 0 && tok < p.vocab) {
                const float s = __fadd_rn(p.score[b], p.logp[static_cast<size_t>(b) * p.logp_stride + tok]);
                if (s != s) {
                    atomicAdd(&n_nan, 1);
                } else {
                    key = (static_cast<uint64_t>(~orderable(s)) << 32) | static_cast<uint32_t>(i);
                    cand_score[i] = s;  // kept for the output (the key's rank drops the sign of -0)
                }
            } else {
                set_status(p.status, SGEMV_ERR_ARG);
                atomicAdd(&n_nan, 1);  // not a candidate
            }
        }
        keys[i] = key;
    }
    __syncthreads();

    // ascending bitonic sort of keys[0, size): the compare-exchange steps of partner distance j >= 32
    // go through shared memory, one CTA barrier each; the steps with j < 32 pair keys of the same warp
    // (key i = tid + m * kBeamThreads is held by lane tid % 32) and run as register shuffles, with one
    // barrier per run of them.
    warp_bitonic(keys, size, tid, 2, 32);  // every step of the lengths 2..32
    for (int len = 64; len <= size; len <<= 1) {
        for (int j = len >> 1; j >= 32; j >>= 1) {
            for (int i = tid; i < size; i += kBeamThreads) {
                const int l = i ^ j;
                if (l > i) {
                    const uint64_t a = keys[i], c = keys[l];
                    const bool up = (i & len) == 0;
                    if ((a > c) == up) {
                        keys[i] = c;
                        keys[l] = a;
                    }
                }
            }
            __syncthreads();
        }
        warp_bitonic(keys, size, tid, len, len);  // the steps j = 16 .. 1 of this length
    }

    const int valid = n - n_nan;
    const int count = valid < p.k ? valid : p.k;
    if (tid < count) {
        const int i = static_cast<int>(keys[tid] & 0xFFFFFFFFu);
        const int b = beam_of(off, p.beam_in, i);
        const int e = first[b] + (i - off[b]);
        const int node = p.child_node[e], tok = p.child_tok[e];
        const float score = cand_score[i];
        p.out_node[tid] = node;
        p.out_score[tid] = score;
        p.out_parent[tid] = b;
        p.out_tok[tid] = tok;
        if (sm.beam_node != nullptr) {
            sm.beam_node[tid] = node;
            sm.beam_score[tid] = score;
            sm.beam_parent[tid] = b;
            sm.beam_tok[tid] = tok;
        }
    }
    if (tid == 0) {
        *p.out_count = count;
        if (n_nan > 0) set_status(p.status, SGEMV_ERR_NONFINITE);
    }
    return count;
}

__global__ void __launch_bounds__(kBeamThreads, 1) beam_step_kernel(const BeamParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ int32_t off[kMaxBeam + 1];
    __shared__ int32_t first[kMaxBeam];
    __shared__ int32_t n_nan;
    // The next step may be scheduled now; everything this step reads may come from the previous kernel
    // in the stream (the previous step's beams, the decoder's scores).
    pdl_launch_dependents();
    pdl_wait();
    StepSmem sm;
    sm.keys = reinterpret_cast<uint64_t*>(smem);
    sm.cand_score = reinterpret_cast<float*>(smem + static_cast<size_t>(p.max_cand) * sizeof(uint64_t));
    sm.off = off;
    sm.first = first;
    sm.n_nan = &n_nan;
    sm.beam_node = nullptr;
    sm.beam_score = nullptr;
    sm.beam_parent = nullptr;
    sm.beam_tok = nullptr;
    beam_step_body(p, sm);
}

// Every step of one decode and the traceback in one launch (the decoder's distributions of all
// positions are known up front, as in the tree-based parallel verification): step t reads its input
// beams from the shared-memory copy of step t-1's output, and the traceback walks the parent links kept
// in shared memory. The per-step outputs and the sequences are also written to global memory.
constexpr int kMaxDecodeSteps = 32;

struct DecodeParams {
    BeamParams step;  // trie, vocab, k, max_cand, status, logp_stride; node, score and beam_in of step 0
    int32_t steps;
    const float* logp[kMaxDecodeSteps];
    int32_t* out_node;    // [steps][k]
    float* out_score;     // [steps][k]
    int32_t* out_parent;  // [steps][k]
    int32_t* out_tok;     // [steps][k]
    int32_t* out_count;   // [steps]
    int32_t* seq;         // [k][steps]
};

__global__ void __launch_bounds__(kBeamThreads, 1) beam_decode_kernel(const __grid_constant__ DecodeParams d) {
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ int32_t off[kMaxBeam + 1];
    __shared__ int32_t first[kMaxBeam];
    __shared__ int32_t n_nan;
    __shared__ int32_t beam_node[2][kMaxBeam];
    __shared__ float beam_score[2][kMaxBeam];
    __shared__ int32_t beam_parent[kMaxDecodeSteps][kMaxBeam];
    __shared__ int32_t beam_tok[kMaxDecodeSteps][kMaxBeam];
    pdl_launch_dependents();
    pdl_wait();  // the first beams and the distributions may come from the previous kernel in the stream
    const int k = d.step.k;
    StepSmem sm;
    sm.keys = reinterpret_cast<uint64_t*>(smem);
    sm.cand_score = reinterpret_cast<float*>(smem + static_cast<size_t>(d.step.max_cand) * sizeof(uint64_t));
    sm.off = off;
    sm.first = first;
    sm.n_nan = &n_nan;
    BeamParams p = d.step;
    int count = 0;
    for (int t = 0; t < d.steps; ++t) {
        if (t > 0) {
            p.node = beam_node[(t - 1) & 1];
            p.score = beam_score[(t - 1) & 1];
            p.beam_in = count;
        }
        p.logp = d.logp[t];
        p.out_node = d.out_node + static_cast<size_t>(t) * k;
        p.out_score = d.out_score + static_cast<size_t>(t) * k;
        p.out_parent = d.out_parent + static_cast<size_t>(t) * k;
        p.out_tok = d.out_tok + static_cast<size_t>(t) * k;
        p.out_count = d.out_count + t;
        sm.beam_node = beam_node[t & 1];
        sm.beam_score = beam_score[t & 1];
        sm.beam_parent = beam_parent[t];
        sm.beam_tok = beam_tok[t];
        count = beam_step_body(p, sm);
        __syncthreads();  // this step's beams and working set are complete before the next step reads them
    }
    const int f = threadIdx.x;  // traceback: seq[f][t] for the final beams f < count, -1 for the others
    if (f < k) {
        int i = f;
        for (int t = d.steps - 1; t >= 0; --t) {
            int tok = -1;
            if (f < count) {
                tok = beam_tok[t][i];
                i = beam_parent[t][i];
            }
            d.seq[static_cast<size_t>(f) * d.steps + t] = tok;
        }
    }
}

// seq[f][t] = token of final beam f at step t, walking the parent links back from the last step.
__global__ void beam_traceback_kernel(int steps, int beam_max, const int32_t* parent, const int32_t* tok,
                                      const int32_t* count, int32_t* seq, int32_t* status) {
    pdl_launch_dependents();
    pdl_wait();  // the last step's outputs come from the previous kernel in the stream
    const int f = blockIdx.x * blockDim.x + threadIdx.x;
    if (f >= beam_max) return;
    const int cnt = *count;
    int i = f;
    for (int t = steps - 1; t >= 0; --t) {
        if (f >= cnt || i < 0 || i >= beam_max) {
            if (f < cnt) set_status(status, SGEMV_ERR_ARG);
            seq[static_cast<size_t>(f) * steps + t] = -1;
            continue;
        }
        seq[static_cast<size_t>(f) * steps + t] = tok[static_cast<size_t>(t) * beam_max + i];
        i = parent[static_cast<size_t>(t) * beam_max + i];
    }
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

}  // namespace sgemv

using namespace sgemv;

extern "C" {

int sgemv_beam_step(const sgemv_trie* trie, int beam_in, int vocab, const int32_t* node_dev,
                    const float* score_dev, const float* logp_dev, int k, int32_t* out_node_dev,
                    float* out_score_dev, int32_t* out_parent_dev, int32_t* out_tok_dev, int32_t* out_count_dev,
                    int32_t* status_dev, void* stream) {
    if (trie == nullptr || trie->child_ptr_dev == nullptr || trie->child_tok_dev == nullptr ||
        trie->child_node_dev == nullptr || trie->n_nodes < 1 || trie->n_edges < 0)
        return SGEMV_ERR_ARG;
    if (beam_in < 1 || beam_in > kMaxBeam || k < 1 || k > kMaxBeam || vocab < 1) return SGEMV_ERR_ARG;
    const void* ptrs[] = {node_dev, score_dev, logp_dev, out_node_dev, out_score_dev, out_parent_dev, out_tok_dev,
                          out_count_dev};
    for (const void* q : ptrs)
        if (q == nullptr) return SGEMV_ERR_ARG;
    for (const void* q : ptrs)
        if (!aligned4(q)) return SGEMV_ERR_ALIGN;
    if (status_dev != nullptr && !aligned4(status_dev)) return SGEMV_ERR_ALIGN;
    BeamParams p;
    p.child_ptr = trie->child_ptr_dev;
    p.child_tok = trie->child_tok_dev;
    p.child_node = trie->child_node_dev;
    p.n_nodes = trie->n_nodes;
    p.n_edges = trie->n_edges;
    p.beam_in = beam_in;
    p.vocab = vocab;
    p.k = k;
    p.node = node_dev;
    p.score = score_dev;
    p.logp = logp_dev;
    p.logp_stride = vocab;
    p.out_node = out_node_dev;
    p.out_score = out_score_dev;
    p.out_parent = out_parent_dev;
    p.out_tok = out_tok_dev;
    p.out_count = out_count_dev;
    p.status = status_dev;
    p.max_cand = kMaxCandidates;
    const int smem = kMaxCandidates * static_cast<int>(sizeof(uint64_t) + sizeof(float));  // keys, scores
    static std::atomic<int> attr_set[64];  // per device: dynamic shared memory already enabled
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SGEMV_ERR_CUDA;
    if (attr_set[dev].load() == 0) {
        if (cudaFuncSetAttribute(beam_step_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return SGEMV_ERR_CUDA;
        attr_set[dev].store(1);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kBeamThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, beam_step_kernel, p) == cudaSuccess ? SGEMV_OK : SGEMV_ERR_CUDA;
}

int sgemv_beam_decode(const sgemv_trie* trie, int steps, int vocab, int beam_in, const int32_t* node_dev,
                      const float* score_dev, const float* const* logp_dev, int logp_stride, int k,
                      int32_t* out_node_dev, float* out_score_dev, int32_t* out_parent_dev, int32_t* out_tok_dev,
                      int32_t* out_count_dev, int32_t* seq_dev, int32_t* status_dev, void* stream) {
    if (trie == nullptr || trie->child_ptr_dev == nullptr || trie->child_tok_dev == nullptr ||
        trie->child_node_dev == nullptr || trie->n_nodes < 1 || trie->n_edges < 0)
        return SGEMV_ERR_ARG;
    if (steps < 1 || steps > kMaxDecodeSteps || beam_in < 1 || beam_in > kMaxBeam || k < 1 || k > kMaxBeam ||
        vocab < 1 || (logp_stride != 0 && logp_stride != vocab) || logp_dev == nullptr)
        return SGEMV_ERR_ARG;
    const void* ptrs[] = {node_dev, score_dev, out_node_dev, out_score_dev, out_parent_dev, out_tok_dev,
                          out_count_dev, seq_dev};
    for (const void* q : ptrs)
        if (q == nullptr) return SGEMV_ERR_ARG;
    for (int t = 0; t < steps; ++t)
        if (logp_dev[t] == nullptr) return SGEMV_ERR_ARG;
    for (const void* q : ptrs)
        if (!aligned4(q)) return SGEMV_ERR_ALIGN;
    for (int t = 0; t < steps; ++t)
        if (!aligned4(logp_dev[t])) return SGEMV_ERR_ALIGN;
    if (status_dev != nullptr && !aligned4(status_dev)) return SGEMV_ERR_ALIGN;
    DecodeParams d;
    std::memset(&d, 0, sizeof(d));
    BeamParams& p = d.step;
    p.child_ptr = trie->child_ptr_dev;
    p.child_tok = trie->child_tok_dev;
    p.child_node = trie->child_node_dev;
    p.n_nodes = trie->n_nodes;
    p.n_edges = trie->n_edges;
    p.beam_in = beam_in;
    p.vocab = vocab;
    p.k = k;
    p.node = node_dev;
    p.score = score_dev;
    p.logp_stride = logp_stride;
    p.status = status_dev;
    p.max_cand = kMaxCandidates;
    d.steps = steps;
    for (int t = 0; t < steps; ++t) d.logp[t] = logp_dev[t];
    d.out_node = out_node_dev;
    d.out_score = out_score_dev;
    d.out_parent = out_parent_dev;
    d.out_tok = out_tok_dev;
    d.out_count = out_count_dev;
    d.seq = seq_dev;
    const int smem = kMaxCandidates * static_cast<int>(sizeof(uint64_t) + sizeof(float));  // keys, scores
    static std::atomic<int> attr_set[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return SGEMV_ERR_CUDA;
    if (attr_set[dev].load() == 0) {
        if (cudaFuncSetAttribute(beam_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return SGEMV_ERR_CUDA;
        attr_set[dev].store(1);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kBeamThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, beam_decode_kernel, d) == cudaSuccess ? SGEMV_OK : SGEMV_ERR_CUDA;
}

int sgemv_beam_traceback(int steps, int beam_max, const int32_t* parent_dev, const int32_t* tok_dev,
                         const int32_t* count_dev, int32_t* seq_dev, int32_t* status_dev, void* stream) {
    if (steps < 1 || beam_max < 1 || beam_max > kMaxBeam) return SGEMV_ERR_ARG;
    if (parent_dev == nullptr || tok_dev == nullptr || count_dev == nullptr || seq_dev == nullptr)
        return SGEMV_ERR_ARG;
    if (!aligned4(parent_dev) || !aligned4(tok_dev) || !aligned4(count_dev) || !aligned4(seq_dev) ||
        (status_dev != nullptr && !aligned4(status_dev)))
        return SGEMV_ERR_ALIGN;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kMaxBeam);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, beam_traceback_kernel, steps, beam_max, parent_dev, tok_dev, count_dev, seq_dev,
                              status_dev) == cudaSuccess
               ? SGEMV_OK
               : SGEMV_ERR_CUDA;
}

}  // extern "C"
