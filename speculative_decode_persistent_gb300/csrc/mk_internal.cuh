// Internal structures of the mk library: the packed weight layout, the model
// and step descriptors the persistent kernel reads, the shared-memory map and
// the static work schedule of the skinny Q4 GEMM phases. Host and device code
// of the library include it; nothing outside csrc/ does.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

#include "mk.h"

namespace mk {

// ------------------------------------------------------------------ launch
constexpr int kWarps = 8;                      // math warps
constexpr int kThreads = kWarps * 32;           // math threads (named barrier 1)
constexpr int kLaunchThreads = kThreads + 32;   // + one producer warp streaming weights

// ------------------------------------------------------------- Q4 "units"
// The GEMM phases stream weights as units of 32 output rows x 256 k
// (one super-block column): 32 row headers of 16 bytes (binary16 d, binary16
// dmin, the 12-byte 6-bit scale/min field, as in the canonical file), then
// 4096 bytes of codes laid out so that each lane of a warp fetches, with one
// 16-byte shared-memory load per sub-block, exactly the nibbles of its
// m16n8k16 A fragments for both 16-row halves and both k-steps.
constexpr int kUnitBytes = 4608;
constexpr int kUnitHdr = 512;
constexpr int kTileRows = 32;

// Per-warp ring of streamed units (bulk async copies, mbarrier completion).
constexpr int kRing = 4;

// ----------------------------------------------------------- shared memory
constexpr int kRingBytes = kWarps * kRing * kUnitBytes;   // 147456
constexpr int kScaleTab = 2048;  // [j8][g8][rb2][hi2] fp32 scales (1 KB); 2 KB as the flush stage
constexpr int kWarpTab = kScaleTab + 128;                 // 2176 per buffer
constexpr int kTabBytes = kWarps * 2 * kWarpTab;          // 34816 (double-buffered per warp)
constexpr int kActBytes = 44 * 1024;                      // activations / phase scratch
constexpr int kMiscBytes = 4096;
constexpr int kBarBytes = 2 * kWarps * kRing * 8;  // full + empty barriers

constexpr int kOffRing = 0;
constexpr int kOffTab = kOffRing + kRingBytes;
constexpr int kOffAct = kOffTab + kTabBytes;
constexpr int kOffMisc = kOffAct + kActBytes;
constexpr int kOffBar = kOffMisc + kMiscBytes;
constexpr int kSmemBytes = kOffBar + kBarBytes;           // 231936
static_assert(kSmemBytes + 256 <= 232448, "exceeds the 227 KB per-block limit");
// Attention and Gated DeltaNet phases may use the table and activation
// regions together (they never hold a GEMM's data at that time).
constexpr int kOffPhase = kOffTab;
constexpr int kPhaseBytes = kTabBytes + kActBytes;        // 79872

// --------------------------------------------------------------- limits
constexpr int kMaxRows = MK_MAX_DECODE_ROWS;  // 12: at most 3 column tiles of 8
constexpr int kMaxT = MK_MAX_T;
constexpr int kMaxSeqs = MK_MAX_SEQS;
constexpr int kMaxDh = 256;
constexpr int kMaxQRows = 48;                 // T x (hq/hkv) rows attending one kv head
constexpr int kMaxSplits = 128;               // split-K parts of one (sequence, kv head)
constexpr int kChunk = 16;                    // cached tokens per attention chunk (one KV page)
constexpr int kAttnMaxSlots = 16;             // KV staging slots (their mbarriers live in misc)
constexpr int kAttnBarOff = 3840;             // byte offset of those mbarriers inside misc
// The page ids of a block's attention item, loaded once by the producer at the
// start of the item's KV stream, live at the end of the ring region.
constexpr int kAttnPageList = 512;            // chunks (pages) of one attention item, at most
constexpr int kAttnPageListBytes = kAttnPageList * 4;
constexpr int kMaxDraft = MK_MAX_T - 1;       // MTP drafts per sequence and step
constexpr int kMaxNormSlices = 16;            // reduction slices of an RMSNorm GEMM phase
// the step's own rows plus the draft passes' positions fit one new-rows chunk
static_assert(kMaxT + kMaxDraft - 1 <= kChunk, "draft positions of one step");

// ------------------------------------------------------------- descriptors
// PRO_MTP_IN: the MTP input rows [RMSNorm(h) w_h ; RMSNorm(emb) w_e], already
// normalised by the MTP input phase.
enum Prologue : int32_t { PRO_RMS_X = 0, PRO_GDN_OUT = 1, PRO_FA_OUT = 2, PRO_H = 3, PRO_MTP_IN = 4 };
enum ZeroBuf : int32_t { ZERO_NONE = 0, ZERO_GU = 1, ZERO_YIN = 2 };
// Outputs of one GEMM phase: input projections into yin, residual add into x
// (red.add; the next RMSNorm sums the squares of the full rows itself), gate/up
// pairs into gu (the SwiGLU is applied by the down projection's prologue),
// logits into the per-warp top-1 records.
enum Epilogue : int32_t { EPI_STORE_YIN = 0, EPI_RESID_X = 1, EPI_STORE_GU = 2, EPI_TOP2 = 3 };

struct GemmDesc {
  const uint8_t* w;  // units [n_tiles][nsb]
  int32_t n_tiles, nsb, n_out, pro, epi;
  int32_t dump;      // EPI_TOP2: 1 = copy the logits to the debug buffer (main lm_head)
  const float* gain;  // RMSNorm gain (PRO_RMS_X) or per-head output-norm gain (PRO_GDN_OUT)
  // a buffer a later phase accumulates into, cleared (rows < R) at this phase's start
  int32_t zero_buf;  // ZERO_NONE, ZERO_GU or ZERO_YIN
  int32_t pad2;
};

struct LayerDesc {
  int32_t kind, gdn_i, fa_i, pad;
  GemmDesc in, o, gu, down;
  const float* conv_w;  // [conv_ch][conv_w]
};

struct ModelDesc {
  int32_t n_layers, H, F, V;
  int32_t hq, hkv, dh, hk, hv, dk, dv, cw, conv_ch;
  int32_t n_gdn, n_fa, n_in_max;      // y_in row stride
  int32_t o_stride;                   // o row stride
  int32_t kv_q8, page_tokens, n_pages, max_pages_per_seq, n_slots, max_seqs;
  int32_t grid;                       // blocks of the persistent launch
  float eps;
  // layer[n_layers] is the MTP block when has_mtp
  LayerDesc layer[MK_MAX_LAYERS + 1];
  GemmDesc lm;
  // MTP draft head: W_fc, and lm_head restricted to rows [0, draft_vocab)
  int32_t has_mtp, n_draft, draft_vocab, pad_mtp;
  GemmDesc mtp_fc, mtp_lm;
  const float* mtp_norm_h;  // [H]
  const float* mtp_norm_e;  // [H]
  float* mtp_in;            // [kMaxRows][2H] normalised input rows of a draft pass
  float* mtp_h;             // [kMaxSeqs][H] hidden output of the previous draft pass
  float2* mtp_rope;         // [kMaxSeqs][kMaxDh/2] (cos, sin) at the next pass's position
  int32_t* mtp_row;         // [kMaxSeqs][2] next pass's token and slot (position - cached length)
  const double* inv_freq;   // [kMaxDh/2] rope_base^(-2i/dh)
  const float* final_norm;
  const uint8_t* embed;               // canonical [V][H/256] super-blocks
  // borrowed state
  void* kv_k; void* kv_v; uint16_t* kv_ks; uint16_t* kv_vs;
  float* gdn_state; float* conv_state;
  // scratch
  float* x;          // [kMaxRows][H] residual stream
  float* yin;        // [kMaxRows][n_in_max] input projections
  float* o;          // [kMaxRows][o_stride] mixer outputs
  float* h;          // [kMaxRows][F] SwiGLU output (written only while debug outputs are on)
  float* gu;         // [kMaxRows][2F] gate/up outputs, 16-row blocks of 8 gate + 8 up rows
  float* logits;     // [kMaxRows][V] lm_head outputs of split tiles (summed by red.add)s
  uint32_t* tickets; // per tile
  float* attn_part;  // [attn items][kMaxAttnGroups][part_rows][part_stride]: dims, then m and l (log2 units)
  int32_t part_rows, part_stride;  // query rows of one (sequence, kv head) at most; dh + 4
  uint32_t* attn_tickets;  // per (step sequence, kv head)
  // RMSNorm row sums of a sliced RMSNorm GEMM phase gp: one partial per
  // reduction slice (written by the slice's first block), [gp][kMaxNormSlices][kMaxRows],
  // and per phase the number of slices published (cleared before each launch)
  float* norm_part;
  uint32_t* norm_cnt;
  float* top_val;    // [grid*kWarps][kMaxRows]
  int32_t* top_idx;  // [grid*kWarps][kMaxRows]
  int32_t* page_table;     // [max_seqs][max_pages_per_seq]
  int32_t* out;      // device result block (see kOut*)
  uint32_t* bar;     // [0] arrivals, [1] generation
  int32_t* err;      // [0] error code, [1] non-finite flag, [2] detail
  float* dbg_logits; // optional
  float* dbg_hidden; // optional
  uint64_t* dbg_time;  // optional: [phases + 1] %globaltimer stamps by block 0
};

// Device result block layout.
constexpr int kOutTokens = 0;                  // [kMaxRows]
constexpr int kOutCounts = kMaxRows;           // [kMaxSeqs]
constexpr int kOutArgmax = kMaxRows + kMaxSeqs;  // [kMaxRows]
constexpr int kOutDrafts = kOutArgmax + kMaxRows;  // [kMaxSeqs][kMaxDraft]
constexpr int kOutInts = kOutDrafts + kMaxSeqs * kMaxDraft;

struct StepDesc {
  int32_t R, n_seq, nt;               // rows, sequences, column tiles of 8
  int32_t n_attn_items;
  int32_t row_tok[kMaxRows], row_pos[kMaxRows], row_si[kMaxRows];
  int32_t seq_id[kMaxSeqs], seq_row0[kMaxSeqs], seq_T[kMaxSeqs], seq_len[kMaxSeqs];
  int32_t seq_slot_in[kMaxSeqs], seq_snap_all[kMaxSeqs];
  // 0: verify rows; 1: prompt rows; 2: prompt rows ending the prompt (one token)
  int32_t seq_prompt[kMaxSeqs];
  int32_t seq_slot_out[kMaxSeqs][kMaxT];
  int32_t seq_nsplit[kMaxSeqs], seq_chunks_per_split[kMaxSeqs], seq_item0[kMaxSeqs];
  // attention plan of this step (attn_plan): query n-tiles, warp groups and KV staging slots
  int32_t attn_nq, attn_jw, attn_wpg, attn_ng, attn_spg, attn_nslots;
  int32_t skip_block, skip_barrier;
  uint64_t barrier_timeout_ns;
  float2 rope[kMaxRows][kMaxDh / 2];  // (cos, sin) of position * base^(-2i/dh)
};

// Error codes in err[0] (device side), mapped to mk_status by the host.
enum : int32_t { DEV_OK = 0, DEV_BARRIER_TIMEOUT = 1, DEV_COPY_TIMEOUT = 2, DEV_BAD_STATE = 3 };

// Source rows of one packed phase matrix: up to four canonical matrices
// stacked vertically, or (interleave_gate_up) the FFN gate and up matrices
// interleaved in blocks of 8 rows.
struct PackSrc {
  int32_t n_seg;
  int32_t row_begin[4], row_end[4];
  const uint8_t* src[4];
  int32_t interleave_gate_up;
};

// ------------------------------------------------------ GEMM work schedule
// Every block computes the same schedule for a phase from (tiles, sb, rows,
// grid): the reduction dimension is cut into S slices so that one slice of
// activations (2 fp16 columns per row: high and low halves) fits in the
// activation region; blocks are divided evenly among slices; inside a slice
// the units (tile-major, super-block-minor) are divided evenly among warps.
struct Sched {
  int32_t S, sb_per;
};

__host__ __device__ inline int act_col_stride(int nsb_slice) { return nsb_slice * 512 + 64; }

// ------------------------------------------------ attention KV staging
// One slot holds one 16-token page of one kv head: K then V, each as boxes
// of 16 rows x box_w bytes written by a 2-D tensor copy (128-byte rows with
// the 128-byte swizzle: 16-byte chunk k of row t lands at chunk k ^ (t & 7);
// q8 rows narrower than 128 bytes are unswizzled 64-byte boxes), then for q8
// the K and V block scales of the page ([16][dh/32] binary16 each).
struct AttnSlot {
  int32_t box_w;      // bytes per box row (128, or 64 for unswizzled q8 boxes)
  int32_t nbox;       // boxes per K (and per V)
  int32_t swz;        // 1: 128-byte swizzle
  int32_t v_off, ks_off, vs_off, bytes, tx_bytes;
};

__host__ __device__ inline AttnSlot attn_slot_layout(int dh, int q8) {
  AttnSlot L;
  const int row_bytes = q8 ? dh : 2 * dh;
  L.swz = (row_bytes % 128 == 0) ? 1 : 0;
  L.box_w = L.swz ? 128 : 64;
  L.nbox = row_bytes / L.box_w;
  const int kv = L.nbox * kChunk * L.box_w;  // bytes of K (or V) codes
  L.v_off = kv;
  L.ks_off = 2 * kv;
  L.vs_off = 2 * kv + (q8 ? kChunk * (dh / 32) * 2 : 0);
  const int end = L.vs_off + (q8 ? kChunk * (dh / 32) * 2 : 0);
  L.bytes = (end + 1023) / 1024 * 1024;
  L.tx_bytes = end;
  return L;
}

// Shared memory of the attention phase (the phase region): Q in binary16
// (8 nq rows of dh + 8 halves), the step's own rows as one more slot, the
// groups' score-exchange buffers from attn_xoff on, and a flag word at the end.
__host__ __device__ constexpr int attn_qbytes(int nq, int dh) { return (nq * 8 * (dh + 8) * 2 + 255) / 256 * 256; }
__host__ __device__ inline int attn_xoff(int nq, int dh, int q8) {
  return attn_qbytes(nq, dh) + (attn_slot_layout(dh, q8).tx_bytes + 255) / 256 * 256;
}

// Warp groups of the attention phase. A group of wpg warps takes attn_nu(nq, q8)
// chunks (16 tokens each) per step. Warp dp of a group owns the head dims of
// the 32-dim blocks dp*jw .. dp*jw+jw-1 (jw = dh / 32 / wpg) for every query
// n-tile (8 of the T x hq/hkv rows attending one kv head): it forms those
// dims' share of the scores and adds P V for the same dims, so each K and V
// element is read and converted by one warp and used for every n-tile. The
// softmax of n-tile q is taken by warp q % wpg alone, from the other warps'
// shares, and handed back as binary16 P fragments and rescale factors. jw
// is the largest power of two up to attn_jw(nq) that divides dh / 32 (a
// warp's accumulators: nq x 2 jw m-tiles of 16 dims); the kernel variant is
// chosen by (nq, jw). ng groups take a block's chunks round-robin, each with
// at least two staging slots, and each writes its own partial.
constexpr int kMaxAttnGroups = 8;
__host__ __device__ constexpr int attn_jw(int nq) { return nq <= 1 ? 4 : nq <= 3 ? 2 : 1; }
// (two chunks a step take more registers: not for the q8 variant of three n-tiles)
__host__ __device__ constexpr int attn_nu(int nq, int q8) { return (nq <= 2 || nq == 4 || (nq == 3 && !q8)) ? 2 : 1; }
// exchange area of one group, in bytes: score shares [wpg-1][nu][nq][32]
// float4, P fragments [nq][nu][32] uint2, factors [nq][32] float2, sums
// [nq][4] float2, and the owners' running state [nq][32] float4
__host__ __device__ constexpr int attn_xslab(int wpg, int nq, int q8) {
  return (wpg - 1) * attn_nu(nq, q8) * nq * 512 + nq * attn_nu(nq, q8) * 256 + nq * 256 + nq * 32 + nq * 512;
}

__host__ __device__ inline void attn_plan(int q_rows_max, int dh, int q8, int ring_bytes, int32_t& nq,
                                          int32_t& jw, int32_t& wpg, int32_t& ng, int32_t& spg,
                                          int32_t& nslots) {
  nq = (q_rows_max + 7) / 8;
  const int nblk = dh / 32;
  jw = attn_jw(nq);
  while (nblk % jw) jw /= 2;
  wpg = nblk / jw;
  const AttnSlot L = attn_slot_layout(dh, q8);
  // room for aligning the first slot to 1024 bytes, and for the page list after the slots
  nslots = (ring_bytes - 1024 - kAttnPageListBytes) / L.bytes;
  if (nslots > kAttnMaxSlots) nslots = kAttnMaxSlots;
  ng = kWarps / wpg;
  if (ng > nslots / 2) ng = nslots / 2;
  if (ng > kMaxAttnGroups) ng = kMaxAttnGroups;
  if (ng < 1) ng = 1;
  const int room = kPhaseBytes - 16 - attn_xoff(nq, dh, q8);
  while (ng > 1 && ng * attn_xslab(wpg, nq, q8) > room) --ng;
  if (ng * attn_xslab(wpg, nq, q8) > room) {  // no plan: the step is refused
    spg = nslots = 0;
    return;
  }
  spg = nslots / ng;
  nslots = spg * ng;
}

// Floats of the merge's weights below the attention phase's flag word.
constexpr int kAttnCombineFloats = (kPhaseBytes - 16) / 4;

// Sub-block sums of the activation rows: [super-block][sub-block][kSxStride]
// floats (rows padded to 12, so a math lane reads four rows with one 16-byte load).
constexpr int kSxStride = kMaxRows;

__host__ __device__ inline int act_bytes(int nsb_slice, int R) {
  return 2 * R * act_col_stride(nsb_slice) + nsb_slice * 8 * kSxStride * 4;  // = 1024 R n + 128 R + 384 n
}

__host__ __device__ inline Sched make_sched(int nsb, int R) {
  // largest slice with act_bytes(n, R) = 1024 R n + 128 R + 384 n <= kActBytes
  Sched s;
  int max_sb = (kActBytes - 128 * R) / (1024 * R + 8 * kSxStride * 4);
  if (max_sb < 1) max_sb = 1;
  if (max_sb > nsb) max_sb = nsb;
  s.S = (nsb + max_sb - 1) / max_sb;
  s.sb_per = (nsb + s.S - 1) / s.S;
  return s;
}

__host__ __device__ inline int slice_sb0(const Sched& s, int sl) { return sl * s.sb_per; }
__host__ __device__ inline int slice_nsb(const Sched& s, int nsb, int sl) {
  int b = sl * s.sb_per, e = b + s.sb_per;
  if (e > nsb) e = nsb;
  return e - b;
}
__host__ __device__ inline int slice_cta0(const Sched& s, int grid, int sl) {
  return static_cast<int>(static_cast<uint32_t>(sl) * grid / s.S);
}
__host__ __device__ inline int slice_of_cta(const Sched& s, int grid, int cta) {
  // largest sl with slice_cta0(sl) <= cta
  return static_cast<int>((static_cast<uint32_t>(cta + 1) * s.S - 1) / grid);
}
// Units [u0, u1) of slice-local warp ws out of Ws warps over Us units
// (32-bit: units x warps stays far below 2^32 for every supported shape).
__host__ __device__ inline uint32_t warp_u0(uint32_t Us, uint32_t Ws, uint32_t ws) {
  return ws * Us / Ws;
}
// Slice-local warp whose range holds unit u.
__host__ __device__ inline uint32_t warp_of_unit(uint32_t Us, uint32_t Ws, uint32_t u) {
  return ((u + 1) * Ws - 1) / Us;
}
// Number of warp ranges that hold units [a, b) of a slice. The even split
// gives every warp floor or ceil(Us/Ws) units: with Us < Ws a range holds at
// most one unit, otherwise none is empty.
__host__ __device__ inline uint32_t segments_in(uint32_t Us, uint32_t Ws, uint32_t a, uint32_t b) {
  if (Us < Ws) return b - a;
  return warp_of_unit(Us, Ws, b - 1) - warp_of_unit(Us, Ws, a) + 1;
}

// One math warp's share of a GEMM phase of n_tiles x nsb units at R rows on
// `grid` blocks: its slice of the reduction, and units [u0, u1) of that
// slice (tile-major, super-block-minor).
struct Assign {
  Sched sc;
  int sl, nsb_s, sb0, cta0;
  uint32_t Us, Ws, ws, u0, u1;
};

__host__ __device__ inline Assign assign_units(int n_tiles, int nsb, int R, int grid, int cta, int warp) {
  Assign a;
  a.sc = make_sched(nsb, R);
  a.sl = slice_of_cta(a.sc, grid, cta);
  a.cta0 = slice_cta0(a.sc, grid, a.sl);
  const int cta1 = slice_cta0(a.sc, grid, a.sl + 1);
  a.nsb_s = slice_nsb(a.sc, nsb, a.sl);
  a.sb0 = slice_sb0(a.sc, a.sl);
  a.Us = static_cast<uint32_t>(n_tiles) * a.nsb_s;
  a.Ws = static_cast<uint32_t>(cta1 - a.cta0) * kWarps;
  a.ws = static_cast<uint32_t>(cta - a.cta0) * kWarps + warp;
  a.u0 = warp_u0(a.Us, a.Ws, a.ws);
  a.u1 = warp_u0(a.Us, a.Ws, a.ws + 1);
  return a;
}

// Contributions a split tile's completion ticket waits for (lm_head tiles
// split across warps when its reduction is not sliced): one per warp range
// holding any of its units, over every slice.
__host__ __device__ inline uint32_t tile_arrivals(const Sched& sc, int n_tiles, int nsb, int grid, uint32_t tile) {
  uint32_t na = 0;
  for (int sl = 0; sl < sc.S; ++sl) {
    const uint32_t ns = slice_nsb(sc, nsb, sl);
    const uint32_t Us = static_cast<uint32_t>(n_tiles) * ns;
    const uint32_t Ws = static_cast<uint32_t>(slice_cta0(sc, grid, sl + 1) - slice_cta0(sc, grid, sl)) * kWarps;
    na += segments_in(Us, Ws, tile * ns, tile * ns + ns);
  }
  return na;
}

}  // namespace mk
