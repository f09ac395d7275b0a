/*
 * ar.h -- C-ABI of libar_gb300.so: the sum all-reduce of n ranks' buffers,
 * emulated on one GB300 (sm_103a), the n ranks being n buffers in its HBM.
 *
 * What is computed (all entry points):
 *   Every rank ends with the elementwise sum of all n ranks' buffers
 *   (handbook chapter "多 GPU 与 NCCL", §集合通信, the all-reduce row).
 *   Sums accumulate in fp32 and are rounded once, round-to-nearest-even, to
 *   the payload type ("SGLang JIT custom all-reduce" notes, §4 "求和
 *   (reduce_impl)").  One-shot, two-shot and the LL/LL128 reduce add the
 *   ranks in rank order 0..n-1 starting from +0, so their outputs are
 *   bit-identical to each other and on every rank (same notes, §4, last
 *   paragraph).  The ring adds chunk c in the order c, c+1, ..., c+n-1
 *   (fp32 partials; ar_ring_rounded rounds them at every hop); ar_tree adds
 *   pairwise, level by level, rounding at every level.
 *
 * Conventions shared by every call:
 *   - Pointers named in/out/src/dst/lines are DEVICE pointers owned by the
 *     caller and must be 16-byte aligned (the notes' §2 and §1: 16-byte
 *     vectors; a misaligned pointer returns AR_ERR_ALIGN).  The arrays
 *     `in`, `out`, `lines_in`, `lines_out` are HOST arrays of n_ranks device
 *     pointers; they are copied into the launch, so they may be freed when
 *     the call returns.
 *   - `count` is in elements of the payload type (0 is a no-op).
 *   - In place is allowed: out[r] == in[r].  Otherwise the buffers of
 *     different ranks, and each rank's input and output, must not overlap
 *     (AR_ERR_INVALID).  Inputs may alias each other (they are only read).
 *   - count x element size must not exceed the handle's max_bytes
 *     (AR_ERR_TOO_LARGE): the library is sized once, up front, the way the
 *     pages' custom all-reduce pre-registers a fixed buffer (handbook chapter
 *     "集合通信：NCCL 的算法、协议与推理框架的定制 all-reduce", §练习
 *     exercise 3).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream), never allocate and never synchronize, so they can be
 *     issued inside CUDA graph capture (tested, with replays, for every
 *     all-reduce call but ar_ring_noalloc and ar_allreduce_rmsnorm; the
 *     optional buffers of AR_OPT_PUSH_STAGING,
 *     AR_OPT_REGISTERED and AR_OPT_PERSISTENT are allocated when the option
 *     is set, never in a call).  Host-side argument errors are
 *     returned at once and nothing is launched.  Errors found by a kernel
 *     are sticky in the handle and are returned by ar_status().
 *   - A handle may be used from one host thread at a time.  Its calls share the
 *     handle's device buffers (the ring's partials, the optional staging,
 *     registered and inbox buffers, the status word), so calls of one handle
 *     whose kernels could overlap on the GPU must be ordered: issue them on one
 *     stream, or order the streams with events.  Calls of different handles are
 *     independent.
 *
 * Return codes: AR_OK (0) or a negative AR_ERR_* value; ar_strerror() names it.
 */
#ifndef AR_GB300_H
#define AR_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* ar_stream_t; /* the same type as cudaStream_t */
typedef struct ar_ctx* ar_handle;        /* opaque */

typedef enum { AR_F32 = 0, AR_BF16 = 1, AR_F16 = 2 } ar_dtype;

enum {
    AR_OK = 0,
    AR_ERR_INVALID = -1,      /* bad handle, n, dtype, step 0, NULL or overlapping pointers */
    AR_ERR_ALIGN = -2,        /* a pointer is not 16-byte aligned */
    AR_ERR_TOO_LARGE = -3,    /* count x element size > max_bytes */
    AR_ERR_CUDA = -4,         /* a CUDA runtime call or a launch failed */
    AR_ERR_FLAG_TIMEOUT = -5, /* an LL/LL128 line never showed the expected flag */
    AR_ERR_WAIT_TIMEOUT = -6  /* a kernel's bounded wait for its own bulk copies, or the
                                 persistent ring's wait for a peer's acknowledgement, ran out */
};

/* Which call an ar_traffic_t describes. */
typedef enum {
    AR_OP_NONE = 0,
    AR_OP_ONE_SHOT = 1,
    AR_OP_TWO_SHOT = 2,
    AR_OP_RING = 3,
    AR_OP_LL_PACK = 4,
    AR_OP_LL_UNPACK = 5,
    AR_OP_LL_REDUCE = 6,
    AR_OP_LL128_PACK = 7,
    AR_OP_LL128_UNPACK = 8,
    AR_OP_LL128_REDUCE = 9,
    AR_OP_ALLREDUCE_RMSNORM = 10,
    AR_OP_ONE_SHOT_PUSH = 11,
    AR_OP_ONE_SHOT_COPYIN = 12,
    AR_OP_RING_ROUNDED = 13,
    AR_OP_TREE = 14,
    AR_OP_RING_PERSISTENT = 15,
    AR_OP_RING_CLUSTER = 16,
    AR_OP_TREE_FUSED = 17,
    AR_OP_RING_FUSED = 18,
    AR_OP_RING_ROUNDED_FUSED = 19
} ar_op;

/* Traffic of one call.
 *   link_bytes_per_rank, steps: the pages' model of a real n-GPU run, for
 *     all-reduce calls: one-shot (n-1) S in 1 step, two-shot 2(n-1)/n S in 2
 *     steps, ring 2(n-1) S / n in 2(n-1) steps (handbook "集合通信：NCCL 的
 *     算法、协议…", §算法; "多 GPU 与 NCCL", §ring all-reduce).  They are
 *     per-rank averages over the call's own chunks; every chunk moves once
 *     per step, so they equal the closed forms for any count.  0 for the
 *     LL/LL128 calls (whose reduce counts as 1 step).
 *   hbm_read_bytes / hbm_write_bytes: the bytes the call must move in this
 *     GPU's HBM (algorithmic, not measured).
 *   launches: kernels the call launched (ar_plan: with the default options,
 *     and for the calls that run in pieces -- ar_ring, ar_ring_rounded,
 *     ar_tree, ar_one_shot_push, ar_one_shot_copyin -- one piece). */
typedef struct {
    int op;                  /* ar_op */
    int n_ranks;             /* 1 for the per-buffer LL/LL128 pack/unpack */
    size_t count;            /* elements */
    size_t elem_bytes;       /* 4 or 2 */
    double link_bytes_per_rank;
    int steps;
    int launches;
    uint64_t hbm_read_bytes;
    uint64_t hbm_write_bytes;
} ar_traffic_t;

/* The sticky device-side error of a handle. */
typedef struct {
    int code;                /* AR_OK, AR_ERR_FLAG_TIMEOUT or AR_ERR_WAIT_TIMEOUT */
    int rank;                /* rank whose line lacked the flag (-1: none) */
    uint64_t line;           /* index of the first line found without its flag */
    uint64_t lines_skipped;  /* lines left unconsumed (their outputs untouched) */
} ar_status_info_t;

/* Options for ar_set_option. */
enum {
    AR_OPT_CTAS_PER_SM = 1,  /* cap on CTAs per SM of a launch, 1..1024; 0 (default): 64
                                (many short-lived CTAs; measured best), and one resident
                                wave for the bulk-copy one-shot */
    AR_OPT_SPIN_NS = 2,      /* LL/LL128 bounded wait per line, ns, 1..10^10 (default 10^6) */
    AR_OPT_ONE_SHOT_IMPL = 3,/* 0 auto, 1 vector loads/stores, 2 bulk-copy staging */
    AR_OPT_TIMING = 4,       /* 0 off (default); k in 1..2^20: record a CUDA event pair
                                around each launch, keeping the last k launches.  Setting
                                it creates the events (not a hot-path call); do not time
                                calls that are being captured into a CUDA graph. */
    AR_OPT_TIMING_PAUSE = 5, /* with AR_OPT_TIMING on: 1 stops recording (no event
                                records at all), 0 resumes; a cheap host-side switch,
                                e.g. to sample every k-th pass of a timed loop */
    AR_OPT_AUTO_POLICY = 7,  /* ar_auto's policy: AR_AUTO_MODEL (default) or AR_AUTO_EMULATED */
    AR_OPT_AUTO_ALPHA_NS = 8,/* model: fixed cost per step, ns (default 1500) */
    AR_OPT_AUTO_BETA_MBS = 9,/* model: per-rank link bandwidth, MB/s (default 450000) */
    AR_OPT_AUTO_HANDOFF = 10,/* model: bytes per rank above which the ring is used (the size
                                of a pre-registered buffer; default 8 MiB; 0 = no hand-off) */
    AR_OPT_PUSH_STAGING = 11,/* 1: allocate the staging slots ar_one_shot_push needs
                                (n x n x max_bytes); 0 (default): free them */
    AR_OPT_REGISTERED = 12,  /* 1: allocate the registered buffers ar_one_shot_copyin needs
                                (n x max_bytes); 0 (default): free them */
    AR_OPT_PERSISTENT = 13,  /* 1: allocate the LL128 inboxes ar_ring_persistent needs
                                (two slots per rank, about 4.3 x max_bytes in all);
                                0 (default): free them */
    AR_OPT_ABSENT_RANK = 14, /* failure emulation for ar_ring_persistent and ar_ring_cluster:
                                rank r (0..n-1) never joins, so its neighbours' waits run out after
                                AR_OPT_SPIN_NS and the status reads AR_ERR_FLAG_TIMEOUT or
                                AR_ERR_WAIT_TIMEOUT; -1 (default): every rank takes part */
    AR_OPT_TWO_SHOT_IMPL = 15,/* ar_two_shot's form, same bits and bytes: 1 two launches (the
                                kernel boundary separates the phases); 2 one launch, each CTA
                                gathering the tile it reduced after a CTA barrier; 3 one launch,
                                tiles handed between CTAs by ready flags; 0 (default): 2 */
    AR_OPT_PDL = 6           /* 1 (default): launch with programmatic stream
                                serialization, so a kernel is scheduled while the one
                                before it in the stream drains (each kernel waits for
                                its predecessor before touching memory); 0: plain launches */
};

/* Kernels, as ar_timing reports them. */
typedef enum {
    AR_K_ONE_SHOT = 1,
    AR_K_REDUCE_SCATTER = 2,  /* two-shot phase 1 */
    AR_K_ALL_GATHER = 3,      /* two-shot phase 2 */
    AR_K_RING_RS_STEP = 4,
    AR_K_RING_AG_STEP = 5,
    AR_K_LL_PACK = 6,
    AR_K_LL_UNPACK = 7,
    AR_K_LL_REDUCE = 8,
    AR_K_LL128_PACK = 9,
    AR_K_LL128_UNPACK = 10,
    AR_K_LL128_REDUCE = 11,
    AR_K_ALLREDUCE_RMSNORM = 12,
    AR_K_PUSH = 13,                 /* one-shot push, phase 1 */
    AR_K_PUSH_REDUCE = 14,          /* one-shot push, phase 2 */
    AR_K_RING_RS_STEP_ROUNDED = 15, /* ar_ring_rounded's reduce-scatter step */
    AR_K_TREE_LEVEL = 16,           /* one level of ar_tree */
    AR_K_RING_PERSISTENT = 17,      /* ar_ring_persistent (all steps) */
    AR_K_COPYIN = 18,               /* ar_one_shot_copyin's copy into the registered buffers */
    AR_K_RING_CLUSTER = 19,         /* ar_ring_cluster (all steps) */
    AR_K_TREE_FUSED = 20,           /* ar_tree_fused (all levels) */
    AR_K_RING_FUSED = 21,           /* ar_ring_fused (all steps) */
    AR_K_RING_ROUNDED_FUSED = 22,   /* ar_ring_rounded_fused (all steps) */
    AR_K_TWO_SHOT = 23              /* ar_two_shot in one launch (both phases) */
} ar_kernel;

/* One timing record: `launches` consecutive launches of one kernel within
 * one call (1, or the n-1 steps of a ring phase), the device time between
 * events recorded on the call's stream right before the first and right after
 * the last (cudaEventElapsedTime), and the HBM bytes they must move
 * (algorithmic).  Average launch time = ms / launches. */
typedef struct {
    int kernel;              /* ar_kernel */
    int op;                  /* ar_op of the call that launched it */
    float ms;
    uint64_t hbm_bytes;
    int launches;
} ar_launch_time_t;

/* ---- handle --------------------------------------------------------------- */

/* Create a handle for n_ranks in [2, 16] ranks of at most max_bytes each
 * (max_bytes >= 16), on the calling thread's current CUDA device.  It
 * allocates, once, the ring's fp32 partial-sum scratch (2 x n_ranks x chunk
 * x 4 B, about 4 x max_bytes), the one-launch two-shot's tile flags (about
 * max_bytes / 128 bytes) and a status word, and creates a stream and two
 * events for the ring's two-stream pieces (see ar_ring).  *out is set only
 * on AR_OK.
 * The n-rank bound is the pages' kMaxNumGPU = 16 (custom all-reduce notes,
 * §调用). */
int ar_create(int n_ranks, size_t max_bytes, ar_handle* out);

/* Synchronize the device, then free the handle and its device memory.  An
 * invalid or NULL handle is AR_ERR_INVALID. */
int ar_destroy(ar_handle h);

/* Set one AR_OPT_* option; out-of-range values are AR_ERR_INVALID. */
int ar_set_option(ar_handle h, int option, int64_t value);

/* ---- all-reduce ------------------------------------------------------------- */

/* One-shot: every rank reads all n buffers and reduces locally, in one step
 * (handbook "集合通信：NCCL 的算法、协议…", §算法, one-shot; custom
 * all-reduce notes §1-§5: 16-byte vectors, n loads in flight, fp32 sum in
 * rank order, one rounding, then the store).  Here one kernel reads each
 * 16-byte vector of the n inputs once and writes the rounded sum to all n
 * outputs.  HBM: reads n S, writes n S. */
int ar_one_shot(ar_handle h, const void* const* in, void* const* out, size_t count,
                ar_dtype dt, ar_stream_t stream);

/* Two-shot: reduce-scatter then all-gather (handbook "集合通信：NCCL 的
 * 算法、协议…", §算法, two-shot, with a synchronization between the phases;
 * "多 GPU 与 NCCL", §集合通信: all-reduce = reduce-scatter + all-gather).
 * Chunk r = elements [rC, min((r+1)C, count)) with C = ceil(count/n) rounded
 * up to a whole 16-byte vector.  Phase 1 writes chunk r's rank-order sum to
 * out[r]; phase 2 copies chunk j of out[j] to every other rank.  Three
 * forms (AR_OPT_TWO_SHOT_IMPL): two launches, the kernel boundary separating
 * the phases; one launch (the default), in which the CTA reducing a tile of a
 * chunk gathers that tile itself after a CTA barrier; or one launch in which
 * the CTA reducing a tile publishes a ready flag and another CTA gathers the
 * tile once it sees the flag (bounded by AR_OPT_SPIN_NS; a wait that runs out
 * leaves that tile's outputs on the other ranks untouched and ar_status
 * reports AR_ERR_WAIT_TIMEOUT; its counters and flags live in the handle,
 * about max_bytes / 128 bytes allocated by ar_create).  Bit-identical to
 * ar_one_shot.  HBM: reads (n+1) S, writes n S. */
int ar_two_shot(ar_handle h, const void* const* in, void* const* out, size_t count,
                ar_dtype dt, ar_stream_t stream);

/* Ring: the chunked ring, step by step ("多 GPU 与 NCCL", §ring all-reduce:
 * n-1 reduce-scatter steps, then n-1 all-gather steps).  Chunks as in
 * ar_two_shot.  Reduce-scatter step s = 0..n-2: for every rank r, rank
 * d = r+1 (mod n) adds its chunk c = r-s (mod n) to the partial that r
 * sends; partials stay fp32 in the handle's scratch and the rank completing
 * a chunk rounds it into its output.  All-gather step s: rank r+1 copies
 * chunk r+1-s (mod n) from rank r.  One launch per step, 2(n-1) launches.
 * Chunk c is summed in the order c, c+1, ..., c+n-1.  When a step's partials
 * (4 count bytes) exceed half of the device's L2, every chunk is cut into P
 * pieces (P = those bytes over half of L2, rounded, at most 64) and the ring
 * runs piece by piece -- a piece's reduce-scatter steps, then its all-gather
 * steps, then the next piece -- so one piece's partials stay in L2 between
 * steps (handbook "集合通信：NCCL 的算法、协议…", §算法: a large message cut
 * into blocks and pipelined): 2(n-1) P launches, the same sums and HBM
 * bytes.  When the partials reach a tenth of L2 the pieces run on two
 * streams, twice as many of half the length: even pieces on `stream`, odd
 * ones on a stream the handle owns, forked from `stream` by an event at the
 * start of the call and joined back into it at the end (so the call stays
 * stream-ordered and graph-capturable); a call made while AR_OPT_TIMING
 * records runs on `stream` alone. */
int ar_ring(ar_handle h, const void* const* in, void* const* out, size_t count,
            ar_dtype dt, ar_stream_t stream);

/* One-shot push (custom all-reduce notes, §实现, where it is named beside
 * one-shot pull): every rank first writes its buffer into a staging slot of
 * every peer, then every rank sums its own slots (its own input for its own
 * term) in rank order.  Needs AR_OPT_PUSH_STAGING (AR_ERR_INVALID
 * otherwise).  Same bits as ar_one_shot.  HBM: reads n S + n^2 S, writes
 * n (n-1) S + n S.  Two launches; when the staged bytes, n (n-1) S, exceed
 * half of the device's L2, the buffers are cut into P pieces (those bytes over
 * half of L2, rounded, at most 64), each staged and reduced in turn: 2 P
 * launches, the pieces on two streams as ar_ring's do (twice as many). */
int ar_one_shot_push(ar_handle h, const void* const* in, void* const* out, size_t count, ar_dtype dt,
                     ar_stream_t stream);

/* One-shot with copy-in (custom all-reduce notes, §5 写回: outside graph
 * capture the input is first copied with cudaMemcpyAsync into a
 * pre-registered buffer that the kernel reads, so the output may be the
 * input itself): one copy kernel fills the handle's n registered buffers
 * (the pages use one cudaMemcpyAsync per rank), then the one-shot kernel
 * reads those.  Needs AR_OPT_REGISTERED (AR_ERR_INVALID otherwise).  Same
 * bits as ar_one_shot.  Two launches.  HBM: reads 2 n S, writes 2 n S.
 * When n S exceeds half of the device's L2, the buffers are cut into P
 * pieces (n S over half of L2, rounded, at most 64), each copied and reduced
 * in turn: 2 P launches, the pieces on two streams as ar_ring's do (twice as
 * many). */
int ar_one_shot_copyin(ar_handle h, const void* const* in, void* const* out, size_t count, ar_dtype dt,
                       ar_stream_t stream);

/* The ring of ar_ring with its partials kept in the payload type and rounded
 * at every hop, the way a library whose buffers hold the payload type does it
 * (each step adds the chunk a rank receives to its own copy, "多 GPU 与
 * NCCL", §ring all-reduce): chunk c gets
 *   RN( ... RN( RN(x_c + x_{c+1}) + x_{c+2} ) ... + x_{c+n-1} ).
 * Equal to ar_ring for fp32; for bf16 / fp16 it may differ from it by the
 * hops' roundings.  HBM: reads 2 e N and writes e N per reduce-scatter step,
 * reads and writes e N per all-gather step.  Runs in pieces as ar_ring does,
 * its step data being e count bytes. */
int ar_ring_rounded(ar_handle h, const void* const* in, void* const* out, size_t count, ar_dtype dt,
                    ar_stream_t stream);

/* Pairwise tree all-reduce (recursive doubling; PCIe-IPC blog post,
 * bhfrc.com/news/61376, §3.1 算法骨架): in each of log2(n) levels, rank r and
 * rank r XOR 2^l read each other's data, add, and both keep the sum rounded
 * to the payload type.  Layout and in-place rules as ar_one_shot; the
 * handle's n_ranks must be a power of two (2, 4, 8 or 16), else
 * AR_ERR_INVALID.  Every rank ends with the same bits; for bf16 / fp16 they
 * may differ from one-shot's by the levels' roundings, for fp32 by the order
 * of the adds.  log2(n) launches; HBM per level: n S read, n S written.
 * When a level's output (n S) exceeds half of the device's L2 the buffer is
 * cut into P pieces (P = n S over half of L2, rounded, at most 64), each
 * taken through all levels in turn, so one piece's level output stays in L2
 * for the next level (handbook "集合通信：NCCL 的算法、协议…", §算法: the tree
 * cuts a large message into blocks and pipelines them): log2(n) P launches,
 * same bits; those pieces run on two streams as ar_ring's do (twice as many,
 * half the length). */
int ar_tree(ar_handle h, const void* const* in, void* const* out, size_t count, ar_dtype dt, ar_stream_t stream);

/* The pairwise tree of ar_tree with all log2(n) levels done in registers in
 * one pass: each thread loads the n ranks' values of a 16-byte vector once,
 * applies every level (the same pairs, adds and roundings) and stores the n
 * results.  Same bits as ar_tree; one launch; HBM reads n S, writes n S (the
 * level-by-level form moves log2(n) times that). */
int ar_tree_fused(ar_handle h, const void* const* in, void* const* out, size_t count, ar_dtype dt,
                  ar_stream_t stream);

/* The ring of ar_ring with all 2(n-1) steps done in registers in one pass
 * ("多 GPU 与 NCCL", §ring all-reduce): per element, chunk c's reduce-scatter
 * is the chain x_c + x_{c+1} + ... + x_{c+n-1} (mod n) of binary32 adds, and
 * the all-gather copies its rounded result unchanged, so each thread loads
 * the n ranks' values of a 16-byte vector once, adds them in that order and
 * stores the one rounded result to all n outputs.  Same chunks, order and
 * bits as ar_ring; layout and in-place rules as ar_one_shot; needs no scratch.
 * One launch; HBM reads n S, writes n S. */
int ar_ring_fused(ar_handle h, const void* const* in, void* const* out, size_t count, ar_dtype dt,
                  ar_stream_t stream);

/* ar_ring_rounded in one pass, as ar_ring_fused: the partial is rounded to
 * the payload type after every hop but the last.  Same bits as
 * ar_ring_rounded.  One launch; HBM reads n S, writes n S. */
int ar_ring_rounded_fused(ar_handle h, const void* const* in, void* const* out, size_t count, ar_dtype dt,
                          ar_stream_t stream);

/* The ring of ar_ring in a single (cooperative) launch, each hop carried as
 * LL128 lines: 120 bytes of fp32 words and an 8-byte step flag per 128 bytes
 * (handbook "集合通信：NCCL 的算法、协议…", §协议; "多 GPU 与 NCCL", §ring
 * all-reduce).  A rank's CTAs poll the flags of the lines the previous rank
 * sends instead of waiting for a kernel boundary, and acknowledge each
 * consumed step so that its two inbox slots can be reused.  When the two
 * slots of a step (all ranks' lines) exceed half of L2, each CTA takes its
 * share of every chunk in pieces (that ratio, rounded, at most 64), each
 * piece through all 2(n-1) steps, so that the lines in flight stay in L2;
 * still one launch.  Same bits as
 * ar_ring.  Needs AR_OPT_PERSISTENT (AR_ERR_INVALID otherwise).  Every wait
 * is bounded by AR_OPT_SPIN_NS: a wait that runs out ends the call early,
 * leaves the outputs incomplete and sets the status (ar_status) to
 * AR_ERR_FLAG_TIMEOUT or AR_ERR_WAIT_TIMEOUT.  All of its CTAs must be
 * resident at once: run nothing else on the device at the same time that
 * could hold SMs for longer than AR_OPT_SPIN_NS.  HBM: reads n e N +
 * 2(n-1) 128 L and writes the same, L = the sum over the n chunks of
 * ceil(chunk length / 30). */
int ar_ring_persistent(ar_handle h, const void* const* in, void* const* out, size_t count, ar_dtype dt,
                       ar_stream_t stream);

/* The ring of ar_ring in one launch with the ranks mapped onto the CTAs of a
 * thread-block cluster (cluster size n_ranks, up to 16): a hop is a batch of
 * 128-byte lines of fp32 partials that the sending CTA writes straight into
 * the receiving CTA's shared memory with asynchronous stores counted on the
 * receiving slot's mbarrier (the handbook's Simple protocol shape: data plus
 * a separate completion signal), so the lines never reach L2 or HBM and the
 * receiver waits on one local barrier.  Each cluster owns a slice of every
 * chunk; clusters are independent.  Short batches (8 lines per warp) for
 * small calls, long ones (32 lines) for large.  Same bits as ar_ring.  Needs
 * no optional buffers.  Waits are bounded by AR_OPT_SPIN_NS as in
 * ar_ring_persistent; AR_OPT_ABSENT_RANK applies.  AR_ERR_CUDA if the device
 * cannot run a cluster of n_ranks CTAs.  HBM: reads n S, writes n S. */
int ar_ring_cluster(ar_handle h, const void* const* in, void* const* out, size_t count, ar_dtype dt,
                    ar_stream_t stream);

/* Ring all-reduce for callers that cannot allocate device memory (code that
 * runs where cudaMalloc is not allowed or not wanted: inside a framework that
 * owns the device heap, a memory-capped process, a plugin that is handed only
 * its input and output buffers).  The pages have no counterpart; it is the
 * same computation as ar_ring (same chunks, rotation and fp32 partials, same
 * bits), without a handle.  The partials live in one static 32 MiB device
 * array inside the library, which every GPU that loads the library holds
 * until the process exits; the call itself allocates nothing.
 *   - Size limit: 2 x n_ranks x C fp32 partials must fit in 32 MiB, with C =
 *     ceil(count / n_ranks) rounded up to a 16-byte vector (about 4 Mi
 *     elements in all: 8 MiB of bf16 per rank at n = 8); larger calls
 *     return AR_ERR_TOO_LARGE.
 *   - The first call on a device, with that device current, looks up the
 *     array's device address and the SM count and keeps them; make that
 *     first call before any stream capture.  Only a successful lookup is
 *     kept: a call whose lookup fails returns AR_ERR_CUDA, and the next call
 *     on that device looks up again.
 *   - Every call shares the array and leaves its partials in it; nothing in
 *     it needs to start at zero.  Calls whose kernels overlap on the GPU
 *     race on it: issue them in order on one stream.
 * Arguments and errors otherwise as ar_ring. */
int ar_ring_noalloc(int n_ranks, const void* const* in, void* const* out, size_t count, ar_dtype dt,
                    ar_stream_t stream);

/* ---- all-reduce fused with residual add and RMSNorm --------------------------- */

/* The decode epilogue of a tensor-parallel layer in one launch (handbook
 * "集合通信：NCCL 的算法、协议…", §源码对照, names such a fused all-reduce +
 * RMSNorm kernel; its result here is that of the unfused chain):
 *   a = the all-reduce of in[*] (as ar_one_shot: rank-order fp32 sum, rounded)
 *   r = RN(a + residual)                                   -> residual_out
 *   y = RN(r * 1/sqrt(mean over the row of r^2 + eps) * w) -> norm_out[0..n-1]
 * in, norm_out: host arrays of n_ranks device pointers to [tokens][hidden]
 * row-major payloads; residual, residual_out: [tokens][hidden] (one copy:
 * in tensor parallelism every rank holds the same residual; residual_out may
 * equal residual); weight: [hidden].  hidden must be a whole number of
 * 16-byte vectors and at most 327680 elements of any payload type (r is
 * kept in fp32, in registers and shared memory: a row of that length spread
 * over 8 CTAs is 160 KiB per CTA); eps >= 0.  In place (norm_out[r] == in[r])
 * is allowed; otherwise no output may overlap an input or another output.
 * Each token row is handled by a thread-block cluster of 16 CTAs (8 for many
 * short rows); each warp sends its partial sum of squares to every CTA of the
 * cluster through distributed shared memory.  a and r match the unfused chain bit for
 * bit; y within one payload ulp (the order of the sum of squares is the
 * kernel's).  ar_plan(AR_OP_ALLREDUCE_RMSNORM) omits the weight's H bytes,
 * which ar_traffic includes after a call. */
int ar_allreduce_rmsnorm(ar_handle h, const void* const* in, const void* residual, const void* weight, float eps,
                         void* const* norm_out, void* residual_out, size_t tokens, size_t hidden, ar_dtype dt,
                         ar_stream_t stream);

/* ---- size-based selection --------------------------------------------------- */

enum {
    /* The pages' choice for n real GPUs (handbook "集合通信：NCCL 的算法、协议…",
     * §算法: small messages one-shot, medium two-shot, large ones handed to
     * the ring of NCCL; the α-β model decides between the first two, the
     * one-shot / two-shot crossover being S* = 2 α β / ((n-1)(1 - 2/n)), none
     * at n = 2 (§练习 exercise 2); frameworks hand buffers above a
     * pre-registered size (about 8 MB in vLLM) to NCCL): the fastest of
     * one-shot, two-shot and ring under the α-β model, and the ring above the
     * hand-off size. */
    AR_AUTO_MODEL = 0,
    /* The cheapest on this GPU: one-shot, which moves the fewest HBM bytes
     * (2 n S) in a single launch at every size. */
    AR_AUTO_EMULATED = 1
};

/* Host only: the call (AR_OP_ONE_SHOT, AR_OP_TWO_SHOT or AR_OP_RING) that
 * `policy` picks for n_ranks buffers of bytes_per_rank bytes; alpha_s in
 * seconds, beta in bytes/s, handoff_bytes 0 for none.  AR_ERR_INVALID for a
 * bad n, policy, alpha or beta. */
int ar_select(int policy, int n_ranks, size_t bytes_per_rank, double alpha_s, double beta_bytes_per_s,
              size_t handoff_bytes);

/* All-reduce with the call the handle's policy (AR_OPT_AUTO_*) selects for
 * this size; then exactly that call.  ar_traffic reports the call chosen. */
int ar_auto(ar_handle h, const void* const* in, void* const* out, size_t count, ar_dtype dt,
            ar_stream_t stream);

/* ---- LL / LL128 protocol lines -------------------------------------------- */
/* Handbook "集合通信：NCCL 的算法、协议…", §协议 table: LL puts 4 B of data
 * and a 4 B flag in every 8 B line, LL128 120 B of data and an 8 B flag in
 * every 128 B line; the receiver checks the flag to know the data arrived.
 * Layout (a reading; the pages give no byte positions):
 *   LL line i    : bytes 0..3 = payload word i (fp32 bits), bytes 4..7 = u32 flag
 *   LL128 line k : bytes 0..119 = payload words 30k..30k+29 (zero padding
 *                  past count), bytes 120..127 = u64 flag
 * Payloads are fp32, count = payload elements.  The flag is the step id;
 * step 0 is rejected (zeroed memory would look valid).  A consumer checks
 * each line's flag, re-reading it for at most AR_OPT_SPIN_NS; a line still
 * without its flag is left unconsumed (its output untouched) and the handle
 * records AR_ERR_FLAG_TIMEOUT for ar_status(). */

/* Bytes of LL lines for a payload of payload_bytes: 2 x payload, payload
 * rounded up to whole 4-byte words. */
size_t ar_ll_bytes(size_t payload_bytes);
/* Bytes of LL128 lines for a payload of payload_bytes: 128 x ceil(P / 120). */
size_t ar_ll128_bytes(size_t payload_bytes);

/* Pack count fp32 words of src into count LL lines with flag `step`. */
int ar_ll_pack(ar_handle h, const float* src, void* lines, size_t count, uint32_t step,
               ar_stream_t stream);
/* Check and unpack count LL lines into dst. */
int ar_ll_unpack(ar_handle h, const void* lines, float* dst, size_t count, uint32_t step,
                 ar_stream_t stream);
/* Pack count fp32 words into ceil(count/30) LL128 lines with flag `step`. */
int ar_ll128_pack(ar_handle h, const float* src, void* lines, size_t count, uint64_t step,
                  ar_stream_t stream);
/* Check and unpack ceil(count/30) LL128 lines into count words of dst. */
int ar_ll128_unpack(ar_handle h, const void* lines, float* dst, size_t count, uint64_t step,
                    ar_stream_t stream);

/* The same for all n_ranks buffers of the handle in one launch: src / lines /
 * dst are host arrays of n_ranks device pointers (each checked as in the
 * single-buffer call; sources may alias, destinations may not overlap
 * anything).  Results are those of n single-buffer calls. */
int ar_ll_pack_n(ar_handle h, const float* const* src, void* const* lines, size_t count, uint32_t step,
                 ar_stream_t stream);
int ar_ll_unpack_n(ar_handle h, const void* const* lines, float* const* dst, size_t count, uint32_t step,
                   ar_stream_t stream);
int ar_ll128_pack_n(ar_handle h, const float* const* src, void* const* lines, size_t count, uint64_t step,
                    ar_stream_t stream);
int ar_ll128_unpack_n(ar_handle h, const void* const* lines, float* const* dst, size_t count, uint64_t step,
                      ar_stream_t stream);

/* Flag-checked reduce: a line is consumed when every rank's copy carries
 * `step`; its words are summed in rank order (fp32, from +0) and written to
 * every rank's output line with flag `step`.  lines_in / lines_out: host
 * arrays of n_ranks device pointers (in place allowed).  count = payload
 * elements per rank.  LL128 sums all 30 words of a line, padding included. */
int ar_ll_reduce(ar_handle h, const void* const* lines_in, void* const* lines_out, size_t count,
                 uint32_t step, ar_stream_t stream);
int ar_ll128_reduce(ar_handle h, const void* const* lines_in, void* const* lines_out, size_t count,
                    uint64_t step, ar_stream_t stream);

/* ---- status, accounting, host-only helpers -------------------------------- */

/* Synchronize the device (every stream, so also the calls this handle
 * issued), return the sticky device error (AR_OK if none) and clear it.  Not
 * for the hot path; a call that fails in CUDA returns AR_ERR_CUDA. */
int ar_status(ar_handle h);
/* As ar_status, with the details of the first failure. */
int ar_status_info(ar_handle h, ar_status_info_t* info);

/* Traffic of the last successful call on this handle. */
int ar_traffic(ar_handle h, ar_traffic_t* t);

/* With AR_OPT_TIMING on: wait for the recorded launches to finish, copy up
 * to `max` of them, oldest first, into out[], set *n_out to the number
 * copied, and clear the record.  AR_ERR_INVALID if timing is off. */
int ar_timing(ar_handle h, ar_launch_time_t* out, int max, int* n_out);

/* Host only, no GPU needed: the traffic a call of `op` would have (as
 * ar_traffic reports it after the call).  For the pack / unpack ops n_ranks
 * is the number of buffers (1 for the single-buffer calls). */
int ar_plan(int op, int n_ranks, size_t count, ar_dtype dt, ar_traffic_t* t);

/* Host only, no GPU needed: the code a call would return for these
 * arguments before launching anything.  op AR_OP_ONE_SHOT, AR_OP_TWO_SHOT,
 * AR_OP_RING, AR_OP_ONE_SHOT_PUSH, AR_OP_ONE_SHOT_COPYIN, AR_OP_RING_ROUNDED,
 * AR_OP_TREE and AR_OP_TREE_FUSED (n_ranks a power of two), AR_OP_RING_PERSISTENT, AR_OP_RING_CLUSTER,
 * AR_OP_RING_FUSED, AR_OP_RING_ROUNDED_FUSED,
 * AR_OP_LL_REDUCE, AR_OP_LL128_REDUCE: the multi-rank calls (n_ranks in
 * [2, 16]; the handle's optional buffers are not checked); AR_OP_LL_PACK, AR_OP_LL_UNPACK, AR_OP_LL128_PACK,
 * AR_OP_LL128_UNPACK: the batched pack / unpack calls over n_ranks buffers
 * (in = sources, out = destinations; n_ranks in [1, 16]).  Pointers are
 * compared, never dereferenced.  For the LL ops dt must be AR_F32. */
int ar_check_args(int op, int n_ranks, size_t max_bytes, const void* const* in,
                  void* const* out, size_t count, ar_dtype dt);

/* Static text for a return code. */
const char* ar_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* AR_GB300_H */
