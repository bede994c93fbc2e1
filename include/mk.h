/*
 * mk — one fused speculative-decode verify cycle on a GB300 (sm_103a).
 *
 * What the library computes is the cycle described on the page "Fusing the
 * whole speculative-decoding cycle into one CUDA kernel" (richland.au),
 * section "What shipped": the main model runs over T = 1 + n_draft rows per
 * sequence, lm_head and greedy verification run on the device, the recurrent
 * state is committed only through the accepted token, and the host reads back
 * only the accepted tokens — all in ONE persistent cooperative kernel launch
 * whose phases are separated by a software grid barrier. Every 4-bit weight is
 * read from HBM once per step for all rows of all sequences (page "OpenJet's
 * CUDA megakernel runs 4 coding agents on one RTX 3090", section "Why it
 * matters"). The model is the hybrid decoder those pages name: Gated DeltaNet
 * layers with a constant-size recurrent state and gated full-attention layers
 * over a paged fp16 or q8 KV cache.
 *
 * Conventions for every entry point:
 *  - Pointers marked "device" are CUDA device addresses on the current device;
 *    "host" pointers are ordinary host memory. Sizes are in elements unless
 *    a name ends in _bytes.
 *  - Buffers the caller passes are BORROWED: they must stay allocated until
 *    mk_free. The library owns only its context, small scratch buffers and
 *    pinned readback buffers, all released by mk_free.
 *  - Every function returns an mk_status; nothing throws across the ABI and
 *    no device code traps. A failed call leaves sequence bookkeeping as it
 *    was unless stated otherwise.
 *  - A context is bound to the stream given at creation; calls on one context
 *    must not overlap (the library is not thread-safe per context).
 */
#ifndef MK_H_
#define MK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MK_MAX_LAYERS 64
#define MK_MAX_SEQS 8
#define MK_MAX_DECODE_ROWS 12 /* rows of one step (all sequences) */
#define MK_MAX_T 8            /* rows of one sequence in one step (1 + drafts) */

typedef enum mk_status {
    MK_OK = 0,
    MK_ERR_INVALID = -1,          /* bad argument, layout or row set */
    MK_ERR_NO_PAGES = -2,         /* KV pool exhausted (checked before any device work) */
    MK_ERR_LAUNCH = -3,           /* cooperative launch refused (e.g. SMs busy) */
    MK_ERR_BARRIER_TIMEOUT = -4,  /* a grid barrier or copy wait gave up; context still usable */
    MK_ERR_PENDING = -5,          /* commit on a sequence with no pending step */
    MK_ERR_NONFINITE = -6,        /* a logit was NaN or Inf */
    MK_ERR_CUDA = -7,             /* a CUDA runtime call failed */
    MK_ERR_UNSUPPORTED = -8       /* shape outside what this build handles */
} mk_status;

/* Layer kinds. */
#define MK_LAYER_GDN 0 /* Gated DeltaNet (linear attention with recurrent state) */
#define MK_LAYER_FA 1  /* gated full attention over the paged KV cache */

/* KV element formats. */
#define MK_KV_F16 0 /* binary16 */
#define MK_KV_Q8 1  /* blocks of 32 int8 codes + one binary16 scale (value = scale * code) */

/*
 * Model and pool shape, copied at mk_create.
 * Constraints: hidden, ffn and every projection input width are multiples of
 * 256 (the Q4 super-block); fa_dh and gdn_dk are multiples of 32;
 * gdn_dk == gdn_dv; fa_hq % fa_hkv == 0; gdn_hv % gdn_hk == 0; conv_w == 4;
 * page_tokens == 16; max_seqs <= MK_MAX_SEQS.
 */
typedef struct mk_layout {
    int32_t n_layers, hidden, ffn, vocab;
    int32_t layer_kind[MK_MAX_LAYERS];
    int32_t fa_hq, fa_hkv, fa_dh;
    float rope_base;
    int32_t gdn_hk, gdn_hv, gdn_dk, gdn_dv, conv_w;
    int32_t tied_lm_head;  /* 1: logits use the embedding matrix */
    int32_t has_mtp;       /* 1: the model has a multi-token-prediction (MTP) draft head */
    int32_t draft_vocab;   /* MTP drafts are argmax over vocabulary rows [0, draft_vocab) */
    int32_t kv_dtype;      /* MK_KV_F16 or MK_KV_Q8 */
    int32_t page_tokens;   /* tokens per KV page (16) */
    int32_t n_pages;       /* pages in the pool */
    int32_t max_seqs;      /* sequence slots */
    int32_t max_pages_per_seq;
    int32_t n_state_slots; /* recurrent-state slots per sequence, >= MK_MAX_T + 1 */
    float rms_eps;         /* RMSNorm and L2-norm epsilon (1e-6) */
    int32_t n_draft;       /* MTP: drafts made per verified sequence and step, 1..MK_MAX_T-1 */
} mk_layout;

/* Canonical weights of one layer. Q4 matrices are [rows][k/256] super-blocks
 * of 144 bytes: binary16 d, binary16 dmin, 96-bit field of 6-bit sub-block
 * scales (bit 6j) and mins (bit 48+6j), then 8 x 16 bytes of 4-bit codes
 * (element i of sub-block j: low nibble of byte i for i < 16, high nibble of
 * byte i-16 otherwise); a weight is d*sc_j*q - dmin*m_j. fp32 vectors as named.
 * All device pointers; read only during mk_create. Unused fields are NULL. */
typedef struct mk_layer_weights {
    const float* attn_norm;  /* [hidden] */
    const void* w_qkv;       /* GDN: [2*hk*dk + hv*dv][hidden] Q4 */
    const void* w_z;         /* GDN: [hv*dv][hidden] Q4 (output gate) */
    const void* w_a;         /* GDN: [hv][hidden] Q4 (alpha = sigmoid(a)) */
    const void* w_b;         /* GDN: [hv][hidden] Q4 (beta = sigmoid(b)) */
    const float* conv_w;     /* GDN: [2*hk*dk + hv*dv][conv_w] causal conv taps, last = current */
    const float* o_norm;     /* GDN: [dv] per-head output RMSNorm gain */
    const void* w_q;         /* FA: [hq*dh][hidden] Q4 */
    const void* w_g;         /* FA: [hq*dh][hidden] Q4 (output gate) */
    const void* w_k;         /* FA: [hkv*dh][hidden] Q4 */
    const void* w_v;         /* FA: [hkv*dh][hidden] Q4 */
    const void* w_o;         /* [hidden][hv*dv or hq*dh] Q4 */
    const float* ffn_norm;   /* [hidden] */
    const void* w_gate;      /* [ffn][hidden] Q4 */
    const void* w_up;        /* [ffn][hidden] Q4 */
    const void* w_down;      /* [hidden][ffn] Q4 */
} mk_layer_weights;

/* The MTP draft head (used when has_mtp): m = W_fc [RMSNorm(h) norm_h ;
 * RMSNorm(embed(next token)) norm_e], one gated-attention decoder layer on m
 * (its own KV layer, the last one of the pool), then RMSNorm(m) final_norm
 * and the lm_head rows [0, draft_vocab). */
typedef struct mk_weights {
    const void* embed;       /* [vocab][hidden] Q4 */
    const float* final_norm; /* [hidden] */
    const void* lm_head;     /* [vocab][hidden] Q4, NULL when tied_lm_head */
    mk_layer_weights layers[MK_MAX_LAYERS];
    mk_layer_weights mtp;        /* MTP block: the gated-attention fields */
    const void* mtp_fc;          /* [hidden][2*hidden] Q4 */
    const float* mtp_norm_h;     /* [hidden] */
    const float* mtp_norm_e;     /* [hidden] */
    const float* mtp_final_norm; /* [hidden] */
} mk_weights;

/* Device buffers the caller allocates (sizes from the mk_*_bytes queries). */
typedef struct mk_buffers {
    void* packed;            /* mk_packed_bytes(): written once by mk_create */
    /* KV pool, one attention layer after another (n_kv = number of gated
     * attention layers, plus one for the MTP block when has_mtp):
     *   F16: k, v   = binary16 [n_kv][n_pages][fa_hkv][page_tokens][fa_dh]
     *   Q8 : k, v   = int8 codes, same shape
     *        k_scale, v_scale = binary16 [n_kv][n_pages][fa_hkv][page_tokens][fa_dh/32] */
    void* kv_k;
    void* kv_v;
    void* kv_k_scale;
    void* kv_v_scale;
    /* Recurrent state per sequence slot and state slot:
     *   gdn_state  fp32 [max_seqs][n_state_slots][n_gdn][hv][dv][dk]
     *   conv_state fp32 [max_seqs][n_state_slots][n_gdn][conv_w-1][2*hk*dk+hv*dv]
     * A sequence's committed state lives in one slot (mk_seq_get reports
     * which); a step writes the state after each of its rows into other slots
     * and commit switches the committed slot, so rollback copies nothing. */
    float* gdn_state;
    float* conv_state;
} mk_buffers;

typedef struct mk_ctx mk_ctx;

/* Byte sizes of the caller-allocated buffers; 0 for an invalid layout. */
size_t mk_packed_bytes(const mk_layout* layout);
size_t mk_kv_bytes(const mk_layout* layout);        /* each of kv_k / kv_v */
size_t mk_kv_scale_bytes(const mk_layout* layout);  /* each of k_scale / v_scale (0 for F16) */
size_t mk_gdn_state_bytes(const mk_layout* layout); /* whole gdn_state buffer */
size_t mk_conv_state_bytes(const mk_layout* layout);/* whole conv_state buffer */

/*
 * Passage: page "OpenJet's CUDA megakernel runs 4 coding agents on one RTX
 * 3090", section "Why it matters" (every step reads all the weights once and
 * stacks every active sequence's rows onto that one read), for the model of
 * page "Fusing the whole speculative-decoding cycle into one CUDA kernel",
 * section "What shipped" (64 layers: 48 Gated DeltaNet, 16 gated attention).
 * Create a context: validates the layout, repacks the canonical weights into
 * buffers->packed (tile order for streaming; the canonical tensors may be
 * freed afterwards), and allocates scratch. stream is a cudaStream_t (NULL =
 * legacy default stream). All sequence slots start empty.
 * Errors: MK_ERR_INVALID (layout/pointers), MK_ERR_UNSUPPORTED (shape),
 * MK_ERR_CUDA (allocation or copy failed).
 */
mk_status mk_create(const mk_layout* layout, const mk_weights* weights,
                    const mk_buffers* buffers, void* stream, mk_ctx** out);

/* The end of a context made by mk_create (the pages describe the engine's
 * step, not its teardown: page "Fusing the whole speculative-decoding cycle
 * into one CUDA kernel", section "What shipped").
 * Release the context, its scratch and pinned buffers. Borrowed buffers are
 * untouched. NULL is accepted. */
void mk_free(mk_ctx* ctx);

/*
 * Install sequence seq with `length` cached tokens whose KV lives on the
 * given pages (host array, page i holds positions 16i..16i+15) and whose
 * recurrent state the caller has written into state slot 0. Pages must be
 * free. Clears any pending step of that slot.
 */
mk_status mk_seq_set(mk_ctx* ctx, int32_t seq, int32_t length, const int32_t* pages,
                     int32_t n_pages);

/* Drop a sequence and return its pages to the pool. */
mk_status mk_seq_reset(mk_ctx* ctx, int32_t seq);

/* Committed view of a sequence: length, page table (host array with room for
 * max_pages_per_seq) and the state slot holding its committed recurrent
 * state. Any output pointer may be NULL. */
mk_status mk_seq_get(mk_ctx* ctx, int32_t seq, int32_t* length, int32_t* pages,
                     int32_t* n_pages, int32_t* state_slot);

/*
 * Passage: page "Fusing the whole speculative-decoding cycle into one CUDA
 * kernel", section "What shipped" (one persistent cooperative launch runs
 * the main model over T = 1 + n_draft rows, lm_head and verification on the
 * device), and page "OpenJet's CUDA megakernel runs 4 coding agents on one
 * RTX 3090", section "Why it matters" (all agents' rows in one batch per
 * step, the host reading back only the accepted tokens).
 * One verify step, synchronous on the context's stream.
 * Rows (host arrays of n_rows): rows of one sequence are contiguous, have
 * consecutive positions starting at the sequence's committed length, and
 * carry the last emitted token in the first row and draft tokens after it.
 * row_flags may be NULL (all 0). 0 = verify row; 1 = prompt row (prefill:
 * the rows are taken as given, nothing is verified); 2 = prompt row that
 * ends its prompt (allowed only as a sequence's last row). All rows of a
 * sequence are of one kind, at most MK_MAX_T of them per step (a longer
 * prompt chunk takes several steps); prompt rows are refused with
 * MK_ERR_UNSUPPORTED when the model has an MTP head. A sequence may appear once.
 * Before the launch the library commits any pending step of the sequences in
 * this step (keeping every accepted row) and allocates pages for the new
 * positions: the lowest free page id first, in row order. With an MTP head
 * the last row of each sequence also reserves the positions its draft passes
 * may write (up to its position + n_draft - 1).
 * Outputs (host): out_tokens[n_rows] receives, per sequence in order of
 * first appearance, the accepted drafts followed by the bonus token (the
 * main model's greedy choice after the last accepted row); out_counts[number
 * of sequences] receives a+1 where a is the number of accepted drafts. For a
 * sequence of prompt rows the count is 0, or 1 when its rows end the prompt
 * (the token is the greedy choice after its last row).
 * The step leaves each verified sequence PENDING until mk_commit or its next
 * step; a sequence of prompt rows is committed through its last row at once.
 * Errors: MK_ERR_INVALID, MK_ERR_NO_PAGES (before any device work),
 * MK_ERR_LAUNCH, MK_ERR_BARRIER_TIMEOUT, MK_ERR_NONFINITE, MK_ERR_CUDA.
 * On a device-side error no sequence becomes pending.
 */
mk_status mk_step(mk_ctx* ctx, int32_t n_rows, const int32_t* tokens, const int32_t* positions,
                  const int32_t* seq_ids, const uint8_t* row_flags, int32_t* out_tokens,
                  int32_t* out_counts);

/*
 * The same step split in three for callers that time or overlap the device
 * part: mk_step_prepare does the host work and queues the small parameter
 * upload; mk_step_launch queues the single cooperative kernel (and may be
 * called again to redo the identical step: it is idempotent until
 * mk_step_finish); mk_step_finish reads back the results and synchronises.
 */
mk_status mk_step_prepare(mk_ctx* ctx, int32_t n_rows, const int32_t* tokens,
                          const int32_t* positions, const int32_t* seq_ids,
                          const uint8_t* row_flags);
mk_status mk_step_launch(mk_ctx* ctx);
mk_status mk_step_finish(mk_ctx* ctx, int32_t* out_tokens, int32_t* out_counts);

/*
 * Drafts the MTP head made in the same launch as the last completed step
 * ("Fusing the whole speculative-decoding cycle into one CUDA kernel", section
 * "What shipped": catch-up rows for the accepted tokens, then n_draft draft
 * steps). drafts (host) receives [sequences of that step, in their order]
 * [n_draft]: for each sequence, catch-up over its accepted rows i = 0..a (row
 * i's final hidden state with the embedding of its greedy token, at its
 * position) gives draft 1 from row a; draft j+1 comes from one more pass on
 * draft j and the head's previous hidden output at position p_a + j. They
 * are the drafts of the sequence's next step when it keeps all accepted rows.
 * Errors: MK_ERR_INVALID (no MTP head, or no completed step).
 */
mk_status mk_last_drafts(mk_ctx* ctx, int32_t* drafts);

/*
 * Passage: page "Fusing the whole speculative-decoding cycle into one CUDA
 * kernel", section "What shipped", the model paragraph (the recurrent state
 * is committed only through the surely-accepted token).
 * Keep n_keep[i] rows (1 <= n_keep[i] <= count of its last step) of each
 * pending sequence seq_ids[i]: the length grows by n_keep, the committed state
 * becomes the one after row n_keep-1, and pages wholly beyond the new length
 * return to the pool. Host-only. Errors: MK_ERR_INVALID, MK_ERR_PENDING.
 */
mk_status mk_commit(mk_ctx* ctx, int32_t n, const int32_t* seq_ids, const int32_t* n_keep);

/* Test hooks: device buffers the next steps fill, or NULL to stop.
 * logits fp32 [n_rows][vocab]; hidden fp32 [n_rows][hidden] = residual stream
 * after the last layer. */
mk_status mk_debug_outputs(mk_ctx* ctx, float* logits, float* hidden);

/* Test hook: copy the step's scratch activations to host memory (fp32,
 * row-major, `rows` rows): residual stream x [rows][hidden]; input
 * projections y [rows][*y_stride] (Gated DeltaNet: qkv | z | a | b;
 * attention: q | gate | k | v); mixer output o [rows][*o_stride]; SwiGLU
 * output h [rows][ffn]. They hold the values of the LAST layer of the last
 * step. NULL buffers are skipped; the strides are always reported.
 * Synchronises the context stream. */
mk_status mk_debug_scratch(mk_ctx* ctx, int32_t rows, float* x, float* y, float* o, float* h,
                           int32_t* y_stride, int32_t* o_stride);

/* Test hook: per-phase timeline. When stamps is a device buffer of at least
 * 5*n_layers + 4 uint64 values, every following launch writes the
 * %globaltimer value (ns) at its start and when block 0 leaves the grid
 * barrier closing each phase (embed, then per layer: input GEMM, mixer,
 * o_proj, gate/up, down; then lm_head; then, with an MTP head only, verify:
 * without one the launch ends at verify; the draft passes are not stamped).
 * NULL stops it. */
mk_status mk_debug_timeline(mk_ctx* ctx, uint64_t* stamps);

/* Test hook: the q8 KV codec that the attention phase applies to the step's
 * own K and V rows, on n_blocks blocks of 32 values. Per block: scale
 * d16[b] = binary16 nearest to max|x| / 127 (ties to even), codes
 * q[32 b + i] = round-half-even(x / d16) clamped to [-127, 127] (0 when
 * d16 = 0); the q8 block of the KV cache as the pages' fused kernel stores it
 * (page "Fusing the whole speculative-decoding cycle into one CUDA kernel",
 * section "What shipped", the paged q8 KV of the model paragraph).
 * x, q, d16: device, fp32 / int8 / binary16 bits. stream: a cudaStream_t
 * (NULL = the legacy default stream); the call waits for it.
 * Errors: MK_ERR_INVALID (null buffer, negative count), MK_ERR_CUDA. */
mk_status mk_debug_q8_encode(const float* x, int64_t n_blocks, int8_t* q, uint16_t* d16, void* stream);

/* Device-side timing of the last mk_step_launch in milliseconds (CUDA events
 * on the context stream); negative if unavailable. */
float mk_last_launch_ms(mk_ctx* ctx);

/* Fault injection for the failure-detection test: the given block skips its
 * arrival at grid barrier number `barrier` of the next launch, so every
 * other block's bounded wait expires. -1 disables. barrier_timeout_ns bounds
 * each wait (0 keeps the default of 500 ms). */
mk_status mk_debug_skip_arrival(mk_ctx* ctx, int32_t block, int32_t barrier,
                                uint64_t barrier_timeout_ns);

/* Bytes the last mk_step_prepare copied host->device (step descriptor and
 * page-table rows) and mk_step_finish copied device->host (result block and
 * error words). Either pointer may be NULL. */
mk_status mk_step_io_bytes(mk_ctx* ctx, uint64_t* h2d_bytes, uint64_t* d2h_bytes);

/* Number of grid blocks of the persistent launch (SM count x blocks per SM). */
int32_t mk_grid_blocks(mk_ctx* ctx);

/*
 * Allocation-free step. The pages have no counterpart of this entry point:
 * it is a deployment aid.
 * Some callers cannot allocate device memory at the moment they step: a
 * server that reserved all of the GPU's memory up front for its own pool
 * (a cudaMalloc there fails, or forces the pool to give memory back), an
 * allocator that must not grow or fragment while requests are in flight,
 * or a latency-critical loop in which a cudaMalloc/cudaFree, which can
 * synchronise the whole device, would stall work on other streams. For
 * them this runs the same step as mk_step, with the same arguments, results
 * and bookkeeping, but every piece of per-step device scratch the kernel
 * writes comes from one file-scope device array of 16 MiB that the library
 * holds on each GPU where it is loaded, until the process exits. The call
 * makes no cudaMalloc, cudaFree or other allocating call; the context itself
 * must already exist (mk_create allocates). Like mk_step it returns after
 * the results are on the host.
 *  - Sizes: a context whose worst-case step scratch exceeds 16 MiB is refused
 *    with MK_ERR_UNSUPPORTED before any bookkeeping changes (small models
 *    fit; the 27B-shaped model does not). So is a model with an MTP head.
 *  - The device that is current must be the context's device
 *    (MK_ERR_INVALID otherwise).
 *  - The first call on a device looks up the array's device address with
 *    cudaGetSymbolAddress; make that first call before any stream capture.
 *  - Every call shares the one array and it keeps the previous call's
 *    contents: the call clears the counters that must start at zero itself.
 *    Calls whose work overlaps on the GPU (two contexts or two streams at
 *    once) race on the array and give wrong results; serialise them.
 *  - mk_last_launch_ms and mk_step_io_bytes report this call as they do
 *    mk_step; mk_debug_scratch reads the context's own buffers, which this
 *    call does not write.
 */
mk_status mk_step_static(mk_ctx* ctx, int32_t n_rows, const int32_t* tokens, const int32_t* positions,
                         const int32_t* seq_ids, const uint8_t* row_flags, int32_t* out_tokens,
                         int32_t* out_counts);

/*
 * Test hook, host only (no context, no device work): the split of one GEMM
 * phase of n_tiles tiles x nsb super-blocks at `rows` rows over `grid`
 * blocks, exactly as the kernel computes it. warp_info (host, grid x
 * warps-per-block x 4 int32, block-major) receives per math warp: the first
 * super-block of its slice of the reduction, the slice width, and its unit
 * range [u0, u1) inside the slice (units are tile-major, super-block-minor).
 * tile_arrivals (host, n_tiles int32) receives, per tile, how many partial
 * contributions its completion ticket waits for. Returns the number of math
 * warps per block, or MK_ERR_INVALID.
 */
int32_t mk_debug_gemm_schedule(int32_t n_tiles, int32_t nsb, int32_t rows, int32_t grid,
                               int32_t* warp_info, int32_t* tile_arrivals);
/* Test hook, host only: shared-memory bytes of the activation operand for a
 * slice of nsb_slice super-blocks at `rows` rows (must fit the kernel's
 * activation region). */
int32_t mk_debug_act_bytes(int32_t nsb_slice, int32_t rows);
/* Test hook, host only: the attention plan mk_step_prepare makes when the
 * longest sequence of a step has q_rows_max query rows per kv head
 * (T x hq/hkv, 1..48), for head dim dh and a q8 (1) or fp16 (0) pool. out
 * (host, 12 int32) receives: query n-tiles nq, 32-dim blocks per warp jw,
 * warps per group wpg, groups ng, staging slots per group spg, slots nslots,
 * the exchange areas' offset in the phase region and one group's area
 * (bytes), the phase region, one slot, the weight ring and the page list
 * (bytes). Returns MK_OK, MK_ERR_INVALID (bad argument) or
 * MK_ERR_UNSUPPORTED (no plan fits: the step would be refused). */
mk_status mk_debug_attn_plan(int32_t q_rows_max, int32_t dh, int32_t q8, int32_t* out);
const char* mk_status_str(mk_status status);

#ifdef __cplusplus
}
#endif
#endif /* MK_H_ */
