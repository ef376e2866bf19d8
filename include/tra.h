/*
 * tra.h -- C ABI of libtra.so: tensor-relational-algebra (TRA) execution of one
 * extended EinSum on one NVIDIA GB300 (sm_103a).
 *
 * Source of the operations: "EinDecomp: automatic tensor-parallel
 * decomposition via Einstein summation + tensor relational algebra".
 *   section 2.1  extended EinSum: Z[out] = AGG_{contracted} OP(X[..], Y[..]);
 *                OP any binary scalar function, AGG commutative and associative
 *   section 2.2  tensor relation (key -> sub-tensor), key -> index range,
 *                join, aggregation, repartition, EinSum -> TRA lowering,
 *                partition vector d (matmul: [d_i, d_jX, d_jY, d_k])
 *   section 3.1  task triple (bound, EinSum, inputs); cost model
 *   section 3.2  task count = number of tuples produced by the join
 *
 * Conventions for every entry point
 *   - Return value: 0 on success, a negative TRA_ERR_* code on failure; the
 *     message of the last failure on the calling thread is ein_last_error().
 *   - Device pointers are plain CUDA device addresses owned by the caller; the
 *     library never allocates or frees device memory.  Host pointers (plans,
 *     info structs, arrays of ints) are read or written only during the call.
 *   - Launches are asynchronous on the given stream (0 = legacy default
 *     stream); nothing synchronises except ein_status().
 *   - Plans are immutable after ein_plan and may be executed concurrently on
 *     different streams.
 *
 * Relation layout ("blocked"): a tensor of shape [B1..Br] under d = [D1..Dr]
 * is one contiguous buffer holding its D1*..*Dr sub-tensors in row-major key
 * order; each sub-tensor (shape [B1/D1..Br/Dr]) is row-major over the
 * tensor's own index order.  Key k holds the index range
 * [k_i*B_i/D_i, (k_i+1)*B_i/D_i) in dimension i (section 2.2).  With d all
 * ones this is the plain dense row-major tensor.
 */
#ifndef TRA_H
#define TRA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* tra_stream_t; /* a cudaStream_t */
typedef struct tra_plan* tra_plan_t;      /* opaque, host-owned */

enum {
    TRA_OK = 0,
    TRA_ERR_PARSE = -1,          /* malformed spec or option */
    TRA_ERR_DIVISIBILITY = -2,   /* some D does not divide its extent B (section 2.2) */
    TRA_ERR_SHARED_LABEL_D = -3, /* a label shared by X and Y got two partition counts */
    TRA_ERR_RANK = -4,           /* wrong number of bounds / d entries, rank too large */
    TRA_ERR_UNSUPPORTED = -5,    /* dtype x operator combination or shape not handled */
    TRA_ERR_WORKSPACE = -6,      /* workspace missing or smaller than ein_plan_info's */
    TRA_ERR_CUDA = -7,           /* a CUDA runtime / driver call failed */
    TRA_ERR_TIMEOUT = -8,        /* a bounded device wait gave up (see ein_status) */
    TRA_ERR_ARG = -9,            /* NULL pointer or invalid argument */
    TRA_ERR_BOUNDS = -10         /* check builds only: a kernel skipped an index outside its buffer */
};

#define TRA_MAX_RANK 8
#define TRA_MAX_LABELS 12

/* Plan summary.  All counts are exact integers (section 3.1 / 3.2 with P read
 * as the number of join tuples; costs are counted in elements). */
typedef struct {
    int32_t n_labels;                  /* distinct labels, first-appearance order X then Y */
    char labels[TRA_MAX_LABELS];       /* label characters */
    int64_t bound[TRA_MAX_LABELS];     /* B_l */
    int32_t part[TRA_MAX_LABELS];      /* D_l */
    int64_t sub_extent[TRA_MAX_LABELS];/* b_l = B_l / D_l */
    int32_t role[TRA_MAX_LABELS];      /* 0 batch (X,Y,Z), 1 M (X,Z), 2 N (Y,Z), 3 contracted */
    int32_t rank_x, rank_y, rank_z;    /* rank_y = 0 for a unary EinSum */
    int32_t key_grid_x[TRA_MAX_RANK];  /* D per index position of X */
    int32_t key_grid_y[TRA_MAX_RANK];
    int32_t key_grid_z[TRA_MAX_RANK];
    uint64_t n_tasks;                  /* join tuples = prod over labels of X u Y of D_l */
    uint64_t n_groups;                 /* output keys = prod over Z's labels of D_l */
    uint64_t n_agg;                    /* join tuples per group = prod over contracted D_l */
    uint64_t x_sub, y_sub, z_sub;      /* elements per sub-tensor */
    uint64_t cost_join;                /* n_tasks * (x_sub + y_sub)            (section 3.1) */
    uint64_t cost_agg;                 /* (n_tasks/n_agg) * (n_agg-1) * z_sub  (section 3.1) */
    uint64_t workspace_bytes;          /* device scratch ein_execute needs (0 = none) */
    int32_t in_dtype, out_dtype;       /* 0 = fp32, 1 = bf16 */
    int32_t kernel;                    /* TRA_KERNEL_* chosen for ein_execute */
    /* terms of the cost-model variants (section 4.3 of the EinDecomp page, see tra_cost_model) */
    uint64_t msg_join;                 /* n_tasks * (number of operands): sub-tensors sent to tasks */
    uint64_t msg_agg;                  /* (n_tasks/n_agg) * (n_agg-1): partials sent to be combined */
    uint64_t mem_elems;                /* |Z| + (n_agg > 1 ? n_tasks * z_sub : 0): output + partials */
} tra_plan_info;

enum {
    TRA_KERNEL_SEMIRING_F32 = 1,  /* CUDA-core join+aggregate (register-tiled) */
    TRA_KERNEL_TC_BF16 = 2,       /* tcgen05 / TMEM / TMA BF16 sum-of-products */
    TRA_KERNEL_ROW_REDUCE = 3,    /* unary aggregation over the contracted labels */
    TRA_KERNEL_ELEMENTWISE = 4,   /* join with AGG = none (broadcast operands allowed) */
    TRA_KERNEL_LSE_FACTORED = 5,  /* logsumexp of a sum: max-shifted exp, then sum-of-products */
    TRA_KERNEL_LITERAL = 6,       /* one partial per join tuple, then ordered combine */
    TRA_KERNEL_TC_BF16_PAIR = 7,  /* as TC_BF16, one 256 x 256 tile per cluster of two CTAs */
    TRA_KERNEL_TC_SPLIT3 = 8,     /* split=bf16x3: squared distance / logsumexp on tensor cores */
    TRA_KERNEL_EMPTY = 9,         /* an output label has extent 0: there is nothing to compute */
    TRA_KERNEL_FILL = 10          /* a contracted label has extent 0: every output aggregates an
                                     empty set, i.e. is agg's identity (0 for sum, -inf for max and
                                     lse, +inf for min) times alpha */
};

/* ein_plan -- build the TRA plan of one EinSum under partition vector d
 * (sections 2.2 "EinSum -> TRA" and 3.1 "task triple").  Host only; touches no device.
 *
 * spec:   "<X labels>,<Y labels>-><Z labels>:<op>:<agg>[:option]..."  or the unary
 *         "<X labels>-><Z labels>::<agg>".  Labels are single letters; a label may
 *         not repeat inside one operand.  op in {mul, add, sqdiff, sub, expsub};
 *         agg in {sum, max, min, lse, none}; none requires that no label is
 *         contracted.  Options: in=f32|bf16 (both inputs, default f32),
 *         out=f32|bf16 (default f32), alpha=<float> (scales the aggregated value),
 *         mode=fused|literal (literal materialises one partial per join tuple and
 *         combines them in canonical order), sqdiff=direct|expand (squared distance as
 *         sum (x - y)^2, or as |x|^2 + |y|^2 - 2 x.y with one FFMA per tuple; default expand
 *         for fp32 inputs with a contracted extent K <= 3127, direct otherwise.  The
 *         expansion cancels where points nearly coincide: every 128 x 128 output tile
 *         holding an output below tau * (|x|^2 + |y|^2), tau = 3 sqrt(K) 2^-24 / 1e-5, is
 *         recomputed in the direct form, so results stay within 1e-5 of D relative, down
 *         to D = 0),
 *         tc=pair|single (BF16 sum-of-products on tensor cores: a 256-row tile
 *         shared by a cluster of two CTAs, or a 128-row tile per CTA; default pair
 *         when the output rows are a multiple of 256 and the columns of 128),
 *         tc_n=256|128 (width of the pair tile; by default 256 where the columns
 *         allow, else 128), tc_store=tma|lsu (tensor-core epilogue: TMA stores
 *         through an output tensor map, the default where one fits, or warp stores),
 *         ksplit=auto|off (tensor-core path: by default the tiles of a last, partly
 *         filled wave of the persistent grid have their K loop split into 2-4 runs on
 *         otherwise idle SMs, the partial sums kept in the workspace and added in a fixed
 *         order, so results stay deterministic; a tile cut in two with an fp32 output
 *         written through a tensor map instead has both halves added into the output,
 *         zeroed at the start of the launch, by TMA reduce-add (the same bits in either
 *         order); off keeps one worker per tile),
 *         split=bf16x3|none (fp32 "sqdiff:sum" and "add:lse" only: the squared-distance
 *         expansion |x|^2 + |y|^2 - 2 x.y, or the factored logsumexp
 *         mx + my + log sum e^(x-mx) e^(y-my), with the sum of products on BF16 tensor cores,
 *         each fp32 operand split as hi + lo bf16 and the product taken as
 *         hi.hi + hi.lo + lo.hi; per product the relative error is at most 3 * 2^-16.
 *         The squared distance keeps the expansion's guard with tau = 4.5 sqrt(K) 2^-24 / 1e-5:
 *         marked 128 x 128 tiles are recomputed on CUDA cores in the direct form.
 *         Default none: these semirings run on CUDA cores).
 * bounds: B_l for every distinct label in first-appearance order (X then Y);
 *         n_bounds must equal the number of distinct labels.  0 <= B_l < 2^31; an
 *         extent of 0 gives an empty EinSum (kernel TRA_KERNEL_EMPTY or _FILL: the key
 *         space, task counts and cost terms are still those of the formulas, with
 *         sub-tensors of 0 elements).
 * d:      partition counts per operand index position, X's then Y's (n_d =
 *         rank_x + rank_y).  A label shared by X and Y must get equal counts.
 * out:    receives the plan; release it with ein_plan_destroy.
 * Errors: TRA_ERR_PARSE, TRA_ERR_RANK, TRA_ERR_DIVISIBILITY, TRA_ERR_SHARED_LABEL_D,
 *         TRA_ERR_UNSUPPORTED, TRA_ERR_ARG. */
int ein_plan(const char* spec, const int64_t* bounds, int n_bounds, const int32_t* d, int n_d, tra_plan_t* out);

/* ein_plan_info -- copy the plan summary (key space, task counts, cost terms). */
int ein_plan_info(tra_plan_t plan, tra_plan_info* info);

/* ein_plan_keys -- the join tuples in canonical order: output key row-major, then the
 * contracted labels' key components (first-appearance order) row-major.  Writes
 * n_tasks rows of (rank_x + rank_y + rank_z) int32: X key, Y key, Z key.
 * capacity: number of int32 the buffer holds; TRA_ERR_ARG if too small. */
int ein_plan_keys(tra_plan_t plan, int32_t* xyz_keys, int64_t capacity);

/* ein_execute -- run the plan: join key-matched sub-tensors through op and aggregate
 * with agg (section 2.2).  in0/in1/out are device buffers in the relation layout of
 * the plan's d (in1 = NULL for a unary EinSum); element types per the in=/out=
 * options (in0, in1 may be NULL for an empty plan, out too when the output has no
 * elements).  out may also be pinned host memory that the device can address (a
 * cudaHostAlloc'd buffer under unified addressing): the kernels then store the result
 * straight into host memory over the host link (the tensor-core kernels switch to their
 * warp-store epilogue for that call; their operands stay in device memory, read through
 * TMA tensor maps).  workspace: device scratch of at least info.workspace_bytes (may be NULL
 * when that is 0); it is overwritten.  Asynchronous on stream.  Calls that may overlap
 * on the GPU need separate workspaces.  Tensor-core plans size their workspace at
 * ein_plan for the device current then (partial sums and flags of the K-split tiles,
 * see ksplit); on another device they run without the split when it does not fit.
 * Errors: TRA_ERR_ARG, TRA_ERR_WORKSPACE, TRA_ERR_CUDA (launch failure). */
int ein_execute(tra_plan_t plan, const void* in0, const void* in1, void* out, void* workspace,
                size_t workspace_bytes, tra_stream_t stream);

/* ein_repartition -- section 2.2 repartition: copy a tensor of the given shape from the
 * relation layout under src_d to the relation layout under dst_d (either may be all
 * ones = dense row-major).  elem_bytes in {1,2,4,8}.  src and dst must not overlap.
 * An extent may be 0 (nothing is copied; src and dst may then be NULL).
 * Asynchronous on stream.  Errors: TRA_ERR_RANK, TRA_ERR_DIVISIBILITY, TRA_ERR_ARG,
 * TRA_ERR_CUDA. */
int ein_repartition(int rank, const int64_t* shape, const int32_t* src_d, const int32_t* dst_d, int elem_bytes,
                    const void* src, void* dst, tra_stream_t stream);

/* ein_repartition_cost -- section 3.1 repartition term.  The pages give no formula;
 * this library counts the elements whose owning block changes when blocks are
 * owned by their row-major linear key id: |T| - sum_L |block_L(src) n block_L(dst)|.
 * Host only. */
int ein_repartition_cost(int rank, const int64_t* shape, const int32_t* src_d, const int32_t* dst_d,
                         uint64_t* cost);

/* ein_repartition_messages -- the repartition's number of communication operations, for the
 * latency term of the cost-model variants: the (source block, destination block) pairs that
 * share at least one element and have different linear key ids.  Host only. */
int ein_repartition_messages(int rank, const int64_t* shape, const int32_t* src_d, const int32_t* dst_d,
                             uint64_t* messages);

/* Cost-model variants (section 4.3 of the EinDecomp page, "troubleshooting"), each off at 0:
 *   latency        added per communication operation: a node's msg_join + msg_agg (see
 *                  tra_plan_info) and an edge's repartition messages; penalises many small tasks
 *   min_block      minimum task granularity: every label's block extent B_l / D_l must be at
 *                  least min(min_block, B_l)
 *   mem_limit      memory-aware pruning: a node's mem_elems may not exceed this many elements
 *   mem_weight     memory-aware cost: mem_weight * mem_elems is added to the node's cost
 *   task_multiple  load balance: n_tasks must be a multiple of this (e.g. the device count)
 * Costs stay in elements; latency and mem_weight convert messages and memory into elements. */
typedef struct {
    uint64_t latency;
    int64_t min_block;
    uint64_t mem_limit;
    uint64_t mem_weight;
    int64_t task_multiple;
} tra_cost_model;

/* ein_graph_decompose -- EinDecomp's optimiser (sections 3.1 and 3.2): choose one
 * partition vector per node of an EinGraph so that the summed cost of section 3.1
 * (every node's join + aggregation cost, plus the repartition cost of every edge
 * whose producer output and consumer input are partitioned differently) is small.
 * Host only.
 *
 * Candidates per node: one partition count D_l per distinct label, each a divisor of
 * B_l (a power of two with TRA_DP_POW2), shared labels equal, with
 * p_min <= n_tasks <= p_max (n_tasks = join tuples; the pages' parallelism
 * constraint asks for at least P, usually exactly P: p_min = p_max = P).
 * Dynamic programme in node order: DP[v][d] = cost(v, d) + sum over v's inputs that
 * are nodes u of min over d' (DP[u][d'] + repartition(u's output under d' -> v's
 * input under d)); the last node is the output; the choice is read back from it.
 * Graph inputs (input -1) arrive in whatever partition their consumer asks for.
 * Where a node feeds two consumers the programme counts its subgraph once per
 * consumer and keeps the choice the later consumer made; total_cost is then
 * recounted with every node and edge once.
 *
 * nodes:  n_nodes entries in topological order (an input index names an earlier node).
 * d_out:  receives every node's vector (X's positions then Y's), nodes in order;
 *         n_d_out must equal the sum of the nodes' ranks.
 * model (may be NULL: the pages' base model): the cost-model variants above, applied to
 *         the candidates (min_block, task_multiple, mem_limit) and to every node and edge cost.
 * node_cost (may be NULL): receives per node join + aggregation + the repartition cost
 *         of its input edges under the chosen vectors (with the model's terms).
 * Errors: TRA_ERR_ARG (NULL, bad input index, node order, output/input shape mismatch,
 *         n_d_out), TRA_ERR_PARSE / TRA_ERR_RANK (a node's spec), TRA_ERR_UNSUPPORTED
 *         (a node has no candidate, or more than 65536). */
typedef struct {
    const char* spec;        /* the node's EinSum as for ein_plan (options are ignored) */
    const int64_t* bounds;   /* B_l per distinct label, first-appearance order X then Y */
    int32_t n_bounds;
    int32_t input[2];        /* producing node of X and of Y, or -1 for a graph input */
} tra_graph_node;

typedef struct {
    uint64_t total_cost;     /* nodes + edges under the chosen vectors, each counted once */
    uint64_t dp_cost;        /* the programme's value at the output node */
    uint64_t n_candidates;   /* partition vectors kept after pruning, over all nodes */
} tra_graph_result;

enum { TRA_DP_POW2 = 1 };

int ein_graph_decompose(const tra_graph_node* nodes, int n_nodes, int64_t p_min, int64_t p_max, int flags,
                        const tra_cost_model* model, int32_t* d_out, int n_d_out, uint64_t* node_cost,
                        tra_graph_result* result);

/* ein_attention -- the attention chain of the multi-head-attention EinGraph (section 2.1)
 * fused into one kernel: Scores[h,s,t] = scale * sum_d Q K, L[h,s] = logsumexp_t Scores,
 * Attn = exp(Scores - L), O[s,h,d] = sum_t Attn V -- without writing Scores or Attn
 * (running max / sum over blocks of 128 keys, O rescaled as the max moves).
 *
 * q:     bf16 [h][s][d]  (the relation of Q_proj under d = [1, h, 1]: head-major)
 * k, v:  bf16 [h][t][d]
 * o:     bf16 [s][h][d]  (dense, as the output projection reads it)
 * lse:   fp32 [h][s] receives L (may be NULL)
 * d must be 128; s and t multiples of 128; device buffers 16-byte aligned (lse 4).
 * Asynchronous on stream; no workspace.  The result is the unfused chain's within the BF16
 * bar: P = Attn is rounded to bf16 before the A.V contraction, as the unfused chain's
 * bf16 Attn is, but against the running max rather than the final L.
 * Errors: TRA_ERR_ARG, TRA_ERR_UNSUPPORTED (shape), TRA_ERR_CUDA. */
int ein_attention(int s, int t, int h, int d, float scale, const void* q, const void* k, const void* v, void* o,
                  void* lse, tra_stream_t stream);

/* ein_status -- synchronise the stream, then read and clear the device status word
 * that bounded waits inside the kernels set when they give up.  Returns TRA_OK,
 * TRA_ERR_TIMEOUT or TRA_ERR_CUDA; in a check build (see ein_build_flags) also
 * TRA_ERR_BOUNDS when a kernel found an index outside its buffer (the message names the
 * first check site; the access was skipped, nothing trapped). */
int ein_status(tra_stream_t stream);

/* ein_execute_sqdist_noalloc -- ein_execute for an fp32 squared-distance plan
 * ("...:sqdiff:sum", expanded form) that needs no caller workspace.  The EinDecomp page
 * has no counterpart: this entry point exists for callers that cannot allocate device
 * memory on their path (memory owned by another allocator or a fixed budget, plugins
 * that may not allocate, paths that must not pay for an allocation and the device
 * synchronisation a free implies).  The row / column norms and the expansion guard's
 * words (one per 128 x 128 output tile) go to a fixed 1 MiB device array inside
 * libtra.so that every GPU loading the library holds until process exit.
 * in0/in1/out: as for ein_execute.  The first call on a device (with that device
 * current) looks up the array's device address; make that first call before any
 * stream capture.  The address is cached per device and context, and looked up again
 * when the context has changed (after cudaDeviceReset).  All calls share the array:
 * calls whose kernels may overlap on the GPU (unordered streams) race.  Nothing is
 * allocated; no clearing is needed (every norm and guard word is rewritten before it
 * is read).  A squared-distance plan with an empty range (TRA_KERNEL_EMPTY / _FILL)
 * needs no scratch and runs as under ein_execute.
 * Errors: TRA_ERR_UNSUPPORTED (not an fp32 expanded squared-distance plan),
 * TRA_ERR_WORKSPACE (norms and guard words need more than 1 MiB: use ein_execute),
 * TRA_ERR_ARG, TRA_ERR_CUDA. */
int ein_execute_sqdist_noalloc(tra_plan_t plan, const void* in0, const void* in1, void* out, tra_stream_t stream);

/* ein_selftest_wait_timeout -- test hook for the bounded device waits: launches one
 * thread that waits on an mbarrier nothing arrives on, with the same bounded wait the
 * tensor-core kernel uses, giving up after timeout_ns.  A following ein_status() on
 * the same stream must return TRA_ERR_TIMEOUT; the context stays usable.
 * Errors: TRA_ERR_CUDA (launch failure). */
int ein_selftest_wait_timeout(uint64_t timeout_ns, tra_stream_t stream);

/* ein_probe_fp32 -- measurement aid (the EinDecomp page has no counterpart): the FP32 issue
 * ceiling of the CUDA-core semiring kernels' inner step.  Launches ctas CTAs of 256 threads
 * (two per SM, as the semiring kernels run); each thread keeps the kernels' 8 x 8 register
 * tile and reads operands from shared memory in their staging layout, iters times 32 k, with
 * no global memory traffic inside the timed loop.  kind 0: two FFMA per two tuples (sum of
 * products); 1: FADD, FADD, one 3-input max.f32 (max-plus); 2: one add.rn.f32x2 and one
 * 3-input max (max-plus, packed add).
 * sink:   device, >= ctas * 256 floats (results that keep the loop alive)
 * cycles: device, >= ctas uint64: SM clocks (clock64) of CTA i's loop
 * nanos:  device, >= ctas uint64: the global timer's ns over the same loop
 * tuples_per_cta (host): receives the tuples one CTA evaluates.
 * Tuples per clock per SM = 2 * tuples_per_cta / cycles; the SM clock = cycles / nanos.
 * Asynchronous on stream.  Errors: TRA_ERR_ARG, TRA_ERR_CUDA. */
int ein_probe_fp32(int kind, int iters, int ctas, void* sink, void* cycles, void* nanos, uint64_t* tuples_per_cta,
                   tra_stream_t stream);

/* ein_build_flags -- how this library was built: TRA_BUILD_CHECK is set in the check build
 * (libtra_check.so, compiled with -DTRA_CHECK).  There every plain global load and store of
 * the CUDA-core semiring, reduction, element-wise, split and repartition kernels and the warp
 * stores of the tensor-core epilogue first test the index against the buffer's extent (the
 * plan's tensors, the workspace's regions); an access outside is skipped and recorded for
 * ein_status.  TMA copies need no test: the tensor maps bound them. */
enum { TRA_BUILD_CHECK = 1 };
int ein_build_flags(void);

/* ein_plan_destroy -- release a plan (NULL is ignored). */
void ein_plan_destroy(tra_plan_t plan);

/* ein_last_error -- message of the last failure on this thread ("" if none). */
const char* ein_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* TRA_H */
