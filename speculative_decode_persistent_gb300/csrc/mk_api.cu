// Host side of the mk C ABI: layout checks, the packed-weight plan, scratch,
// the per-sequence bookkeeping (length, page table, committed state slot,
// pending verify result), the page allocator (lowest free page first, in row
// order; pages wholly beyond the committed length are freed), the per-step
// descriptor and the single cooperative launch.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <set>
#include <vector>

#include "mk_internal.cuh"

namespace mk {
cudaError_t pack_units(const PackSrc& p, uint8_t* dst, int n_tiles, int nsb, cudaStream_t s);
cudaError_t launch_persistent(const ModelDesc* md, const StepDesc* sd, int grid,
                              const CUtensorMap* tm_k, const CUtensorMap* tm_v, cudaStream_t stream);
cudaError_t launch_q8_encode(const float* x, int64_t n_blocks, int8_t* q, uint16_t* d16, cudaStream_t stream);
cudaError_t configure_persistent(int* blocks_per_sm);
}  // namespace mk

using namespace mk;

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }
int tiles_of(int rows) { return (rows + kTileRows - 1) / kTileRows; }
size_t q4_bytes(int rows, int k) { return static_cast<size_t>(rows) * (k / 256) * 144; }

struct PhasePlan {
  size_t off = 0;
  int n_tiles = 0, nsb = 0, n_out = 0;
};

struct Plan {
  bool ok = false;
  int n_gdn = 0, n_fa = 0, conv_ch = 0, n_in_gdn = 0, n_in_fa = 0, n_in_max = 0, o_stride = 0;
  // index MK_MAX_LAYERS holds the MTP block
  PhasePlan in[MK_MAX_LAYERS + 1], o[MK_MAX_LAYERS + 1], gu[MK_MAX_LAYERS + 1], down[MK_MAX_LAYERS + 1], lm;
  PhasePlan mtp_fc;
  size_t off_embed = 0;
  size_t off_attn_norm[MK_MAX_LAYERS + 1], off_ffn_norm[MK_MAX_LAYERS + 1], off_conv[MK_MAX_LAYERS],
      off_onorm[MK_MAX_LAYERS], off_final_norm = 0;
  size_t off_mtp_norm_h = 0, off_mtp_norm_e = 0, off_mtp_final_norm = 0;
  size_t total = 0;
};

bool layout_ok(const mk_layout& L) {
  if (L.n_layers < 1 || L.n_layers > MK_MAX_LAYERS) return false;
  if (L.hidden <= 0 || L.hidden % 256 || L.ffn <= 0 || L.ffn % 256 || L.vocab <= 0) return false;
  bool has_fa = false, has_gdn = false;
  for (int l = 0; l < L.n_layers; ++l) {
    if (L.layer_kind[l] == MK_LAYER_FA) has_fa = true;
    else if (L.layer_kind[l] == MK_LAYER_GDN) has_gdn = true;
    else return false;
  }
  if (has_fa || L.has_mtp) {  // the MTP block is a gated-attention layer
    if (L.fa_hq <= 0 || L.fa_hkv <= 0 || L.fa_hq % L.fa_hkv) return false;
    if (L.fa_dh <= 0 || L.fa_dh % 64 || L.fa_dh > kMaxDh) return false;
    if ((L.fa_hq * L.fa_dh) % 256) return false;
    if (L.fa_hq / L.fa_hkv > kMaxQRows) return false;
  }
  if (has_gdn) {
    if (L.gdn_hk <= 0 || L.gdn_hv <= 0 || L.gdn_hv % L.gdn_hk) return false;
    if (L.gdn_dk != L.gdn_dv || L.gdn_dk % 32 || L.gdn_dk > 128) return false;
    if ((L.gdn_hv * L.gdn_dv) % 256) return false;
    if (256 % L.gdn_dv) return false;
    if (L.conv_w != 4) return false;
  }
  if (L.has_mtp) {
    if (L.n_draft < 1 || L.n_draft > kMaxDraft) return false;
    if (L.draft_vocab < 1 || L.draft_vocab > L.vocab) return false;
  }
  if (L.kv_dtype != MK_KV_F16 && L.kv_dtype != MK_KV_Q8) return false;
  if (L.page_tokens != 16 || L.n_pages <= 0) return false;
  if (L.max_seqs <= 0 || L.max_seqs > MK_MAX_SEQS || L.max_pages_per_seq <= 0) return false;
  if (L.n_state_slots < 2) return false;
  if (!(L.rms_eps >= 0.f)) return false;
  // an RMSNorm phase's reduction slices at the most rows must fit the row-sum slots
  if (make_sched(L.hidden / 256, kMaxRows).S > kMaxNormSlices) return false;
  return true;
}

// GEMM phases of one launch: four per layer, lm_head, six per MTP draft pass.
int gemm_phases(const mk_layout& L) { return 4 * L.n_layers + 1 + (L.has_mtp ? 6 * L.n_draft : 0); }

Plan make_plan(const mk_layout& L) {
  Plan p;
  if (!layout_ok(L)) return p;
  const int H = L.hidden, F = L.ffn;
  p.conv_ch = 2 * L.gdn_hk * L.gdn_dk + L.gdn_hv * L.gdn_dv;
  p.n_in_gdn = p.conv_ch + L.gdn_hv * L.gdn_dv + 2 * L.gdn_hv;
  p.n_in_fa = 2 * L.fa_hq * L.fa_dh + 2 * L.fa_hkv * L.fa_dh;
  size_t at = 0;
  auto phase = [&](PhasePlan& ph, int rows, int k) {
    ph.off = at;
    ph.n_tiles = tiles_of(rows);
    ph.nsb = k / 256;
    ph.n_out = rows;
    at = align_up(at + static_cast<size_t>(ph.n_tiles) * ph.nsb * kUnitBytes);
  };
  for (int l = 0; l < L.n_layers; ++l) {
    const bool gdn = L.layer_kind[l] == MK_LAYER_GDN;
    if (gdn) ++p.n_gdn; else ++p.n_fa;
    const int n_in = gdn ? p.n_in_gdn : p.n_in_fa;
    const int k_o = gdn ? L.gdn_hv * L.gdn_dv : L.fa_hq * L.fa_dh;
    p.n_in_max = std::max(p.n_in_max, n_in);
    p.o_stride = std::max(p.o_stride, k_o);
    phase(p.in[l], n_in, H);
    phase(p.o[l], H, k_o);
    phase(p.gu[l], 2 * F, H);
    phase(p.down[l], H, F);
  }
  phase(p.lm, L.vocab, H);
  if (L.has_mtp) {
    const int M = MK_MAX_LAYERS;
    phase(p.mtp_fc, H, 2 * H);
    phase(p.in[M], p.n_in_fa, H);
    phase(p.o[M], H, L.fa_hq * L.fa_dh);
    phase(p.gu[M], 2 * F, H);
    phase(p.down[M], H, F);
    p.n_in_max = std::max(p.n_in_max, p.n_in_fa);
    p.o_stride = std::max(p.o_stride, L.fa_hq * L.fa_dh);
  }
  p.n_in_max = tiles_of(p.n_in_max) * kTileRows;
  p.off_embed = at;
  at = align_up(at + q4_bytes(L.vocab, H));
  for (int l = 0; l < L.n_layers; ++l) {
    p.off_attn_norm[l] = at; at = align_up(at + H * 4);
    p.off_ffn_norm[l] = at; at = align_up(at + H * 4);
    if (L.layer_kind[l] == MK_LAYER_GDN) {
      p.off_conv[l] = at; at = align_up(at + static_cast<size_t>(p.conv_ch) * 4 * 4);
      p.off_onorm[l] = at; at = align_up(at + L.gdn_dv * 4);
    }
  }
  p.off_final_norm = at;
  at = align_up(at + H * 4);
  if (L.has_mtp) {
    const int M = MK_MAX_LAYERS;
    p.off_attn_norm[M] = at; at = align_up(at + H * 4);
    p.off_ffn_norm[M] = at; at = align_up(at + H * 4);
    p.off_mtp_norm_h = at; at = align_up(at + H * 4);
    p.off_mtp_norm_e = at; at = align_up(at + H * 4);
    p.off_mtp_final_norm = at; at = align_up(at + H * 4);
  }
  p.total = at;
  p.ok = true;
  return p;
}

struct SeqInfo {
  bool used = false;
  int len = 0;
  std::vector<int> pages;
  int slot = 0;
  bool pending = false;
  int count = 0;
  int snap_slot[kMaxT] = {0};
};

}  // namespace

struct mk_ctx {
  mk_layout L;
  std::vector<int32_t> drafts;  // [sequences of the last completed step][n_draft]
  Plan plan;
  cudaStream_t stream = nullptr;
  int device = 0;  // the device current at mk_create
  int grid = 0;
  ModelDesc md_host;
  ModelDesc* md_dev = nullptr;
  StepDesc* sd_dev = nullptr;
  StepDesc* sd_host = nullptr;  // pinned
  int32_t* out_host = nullptr;  // pinned [kOutInts + 4]
  int32_t* pt_host = nullptr;   // pinned page-table mirror
  double* inv_freq = nullptr;  // device [kMaxDh/2]
  CUtensorMap tm_k{}, tm_v{};  // 2-D tensor maps of the K and V pools (attention page copies)
  std::vector<void*> allocs;
  std::vector<SeqInfo> seqs;
  std::set<int> free_pages;
  cudaEvent_t ev0 = nullptr, ev1 = nullptr;
  bool timed = false;
  // prepared step
  bool prepared = false;
  bool launched = false;
  int n_rows = 0, n_seq = 0;
  int step_seq[kMaxSeqs];
  int step_T[kMaxSeqs];
  int step_snap[kMaxSeqs][kMaxT];
  int step_prompt[kMaxSeqs];  // 0 verify, 1 prompt rows, 2 prompt rows ending the prompt
  int skip_block = -1, skip_barrier = -1;
  uint64_t barrier_timeout_ns = 500000000ull;
  size_t tickets_bytes = 0, attn_tickets_bytes = 0;
  uint64_t h2d_bytes = 0, d2h_bytes = 0;
};

namespace {

template <typename T>
cudaError_t dev_alloc(mk_ctx* c, T** p, size_t bytes) {
  void* v = nullptr;
  cudaError_t e = cudaMalloc(&v, bytes ? bytes : 16);
  if (e != cudaSuccess) return e;
  c->allocs.push_back(v);
  *p = static_cast<T*>(v);
  return cudaMemsetAsync(v, 0, bytes ? bytes : 16, c->stream);
}

void release_pages(mk_ctx* c, SeqInfo& s) {
  const int need = (s.len + c->L.page_tokens - 1) / c->L.page_tokens;
  while (static_cast<int>(s.pages.size()) > need) {
    c->free_pages.insert(s.pages.back());
    s.pages.pop_back();
  }
}

void commit_seq(mk_ctx* c, SeqInfo& s, int keep) {
  s.len += keep;
  s.slot = s.snap_slot[keep - 1];
  s.pending = false;
  release_pages(c, s);
}

cudaError_t upload_pages(mk_ctx* c, int seq) {
  const SeqInfo& s = c->seqs[seq];
  int32_t* row = c->pt_host + static_cast<size_t>(seq) * c->L.max_pages_per_seq;
  for (size_t i = 0; i < s.pages.size(); ++i) row[i] = s.pages[i];
  if (s.pages.empty()) return cudaSuccess;
  c->h2d_bytes += s.pages.size() * sizeof(int32_t);
  return cudaMemcpyAsync(c->md_host.page_table + static_cast<size_t>(seq) * c->L.max_pages_per_seq, row,
                         s.pages.size() * sizeof(int32_t), cudaMemcpyHostToDevice, c->stream);
}

// Bookkeeping of a completed step from the result block h: verified
// sequences become pending with their accepted count (mk_commit or the next
// step commits); prompt rows are committed through their last row at once.
// False when the device reported an impossible count.
bool finish_seqs(mk_ctx* c, const int32_t* h, int32_t* out_tokens, int32_t* out_counts) {
  // every count is checked before any sequence changes, so an impossible
  // result block leaves the bookkeeping as it was
  for (int i = 0; i < c->n_seq; ++i) {
    const int cnt = h[kOutCounts + i];
    if (c->step_prompt[i] ? cnt != (c->step_prompt[i] == 2 ? 1 : 0) : (cnt < 1 || cnt > c->step_T[i])) return false;
  }
  int at = 0;
  for (int i = 0; i < c->n_seq; ++i) {
    const int cnt = h[kOutCounts + i];
    const int T = c->step_T[i];
    SeqInfo& s = c->seqs[c->step_seq[i]];
    for (int t = 0; t < T; ++t) s.snap_slot[t] = c->step_snap[i][t];
    s.pending = true;
    if (c->step_prompt[i]) {
      s.count = T;
      commit_seq(c, s, T);
    } else {
      s.count = cnt;
    }
    if (out_counts) out_counts[i] = cnt;
    for (int k = 0; k < cnt; ++k) {
      if (out_tokens) out_tokens[at] = h[kOutTokens + at];
      ++at;
    }
  }
  return true;
}

}  // namespace

extern "C" {

size_t mk_packed_bytes(const mk_layout* layout) {
  if (!layout) return 0;
  const Plan p = make_plan(*layout);
  return p.ok ? p.total : 0;
}

static int n_fa_of(const mk_layout* L) {
  int n = 0;
  for (int l = 0; l < L->n_layers && l < MK_MAX_LAYERS; ++l) n += L->layer_kind[l] == MK_LAYER_FA;
  return n;
}

// KV layers of the pool: one per gated-attention layer, plus the MTP block's.
static int n_kv_of(const mk_layout* L) { return n_fa_of(L) + (L->has_mtp ? 1 : 0); }

size_t mk_kv_bytes(const mk_layout* L) {
  if (!L || !layout_ok(*L)) return 0;
  const size_t elems = static_cast<size_t>(n_kv_of(L)) * L->n_pages * L->fa_hkv * L->page_tokens * L->fa_dh;
  return elems * (L->kv_dtype == MK_KV_Q8 ? 1 : 2);
}

size_t mk_kv_scale_bytes(const mk_layout* L) {
  if (!L || !layout_ok(*L) || L->kv_dtype != MK_KV_Q8) return 0;
  return static_cast<size_t>(n_kv_of(L)) * L->n_pages * L->fa_hkv * L->page_tokens * (L->fa_dh / 32) * 2;
}

size_t mk_gdn_state_bytes(const mk_layout* L) {
  if (!L || !layout_ok(*L)) return 0;
  const size_t n_gdn = L->n_layers - n_fa_of(L);
  return static_cast<size_t>(L->max_seqs) * L->n_state_slots * n_gdn * L->gdn_hv * L->gdn_dv * L->gdn_dk * 4;
}

size_t mk_conv_state_bytes(const mk_layout* L) {
  if (!L || !layout_ok(*L)) return 0;
  const size_t n_gdn = L->n_layers - n_fa_of(L);
  const size_t C = 2 * L->gdn_hk * L->gdn_dk + L->gdn_hv * L->gdn_dv;
  return static_cast<size_t>(L->max_seqs) * L->n_state_slots * n_gdn * (L->conv_w - 1) * C * 4;
}

const char* mk_status_str(mk_status s) {
  switch (s) {
    case MK_OK: return "ok";
    case MK_ERR_INVALID: return "invalid argument";
    case MK_ERR_NO_PAGES: return "KV page pool exhausted";
    case MK_ERR_LAUNCH: return "cooperative launch refused";
    case MK_ERR_BARRIER_TIMEOUT: return "grid barrier or copy wait timed out";
    case MK_ERR_PENDING: return "no pending step on this sequence";
    case MK_ERR_NONFINITE: return "non-finite logits";
    case MK_ERR_CUDA: return "CUDA runtime error";
    case MK_ERR_UNSUPPORTED: return "unsupported shape";
  }
  return "unknown status";
}

void mk_free(mk_ctx* c) {
  if (!c) return;
  cudaStreamSynchronize(c->stream);
  for (void* p : c->allocs) cudaFree(p);
  if (c->sd_host) cudaFreeHost(c->sd_host);
  if (c->out_host) cudaFreeHost(c->out_host);
  if (c->pt_host) cudaFreeHost(c->pt_host);
  if (c->ev0) cudaEventDestroy(c->ev0);
  if (c->ev1) cudaEventDestroy(c->ev1);
  delete c;
}

// 2-D tensor map over one KV pool: rows = (attention layer, page, kv head,
// token), columns = the head's dh elements; boxes of 16 rows x box_w bytes.
bool encode_kv_map(CUtensorMap* m, void* base, const mk_layout& L, int n_fa) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return false;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const int q8 = L.kv_dtype == MK_KV_Q8;
  const AttnSlot S = attn_slot_layout(L.fa_dh, q8);
  const int esz = q8 ? 1 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(L.fa_dh),
                        static_cast<cuuint64_t>(n_fa) * L.n_pages * L.fa_hkv * L.page_tokens};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(L.fa_dh) * esz};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(S.box_w / esz), static_cast<cuuint32_t>(kChunk)};
  cuuint32_t estr[2] = {1, 1};
  return encode(m, q8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, base, dims, strides,
                box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                S.swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

mk_status mk_create(const mk_layout* layout, const mk_weights* w, const mk_buffers* b, void* stream,
                    mk_ctx** out) {
  if (!layout || !w || !b || !out) return MK_ERR_INVALID;
  *out = nullptr;
  if (!layout_ok(*layout)) return MK_ERR_UNSUPPORTED;
  const mk_layout& L = *layout;
  if (!b->packed || !b->kv_k || !b->kv_v || !b->gdn_state || !b->conv_state) return MK_ERR_INVALID;
  if (L.kv_dtype == MK_KV_Q8 && (!b->kv_k_scale || !b->kv_v_scale)) return MK_ERR_INVALID;
  if (!w->embed || !w->final_norm || (!L.tied_lm_head && !w->lm_head)) return MK_ERR_INVALID;
  mk_ctx* c = new (std::nothrow) mk_ctx();
  if (!c) return MK_ERR_CUDA;
  c->L = L;
  c->stream = static_cast<cudaStream_t>(stream);
  c->plan = make_plan(L);
  const Plan& p = c->plan;
  uint8_t* packed = static_cast<uint8_t*>(b->packed);
  const int H = L.hidden, F = L.ffn;

  // ---- repack weights
  auto pack = [&](const PhasePlan& ph, PackSrc src) -> bool {
    return pack_units(src, packed + ph.off, ph.n_tiles, ph.nsb, c->stream) == cudaSuccess;
  };
  bool ok = true;
  for (int l = 0; l < L.n_layers && ok; ++l) {
    const mk_layer_weights& lw = w->layers[l];
    const bool gdn = L.layer_kind[l] == MK_LAYER_GDN;
    PackSrc s{};
    if (gdn) {
      if (!lw.w_qkv || !lw.w_z || !lw.w_a || !lw.w_b || !lw.conv_w || !lw.o_norm) { ok = false; break; }
      const int C = p.conv_ch, vd = L.gdn_hv * L.gdn_dv, hv = L.gdn_hv;
      s.n_seg = 4;
      s.row_begin[0] = 0; s.row_end[0] = C; s.src[0] = static_cast<const uint8_t*>(lw.w_qkv);
      s.row_begin[1] = C; s.row_end[1] = C + vd; s.src[1] = static_cast<const uint8_t*>(lw.w_z);
      s.row_begin[2] = C + vd; s.row_end[2] = C + vd + hv; s.src[2] = static_cast<const uint8_t*>(lw.w_a);
      s.row_begin[3] = C + vd + hv; s.row_end[3] = C + vd + 2 * hv; s.src[3] = static_cast<const uint8_t*>(lw.w_b);
    } else {
      if (!lw.w_q || !lw.w_g || !lw.w_k || !lw.w_v) { ok = false; break; }
      const int qd = L.fa_hq * L.fa_dh, kd = L.fa_hkv * L.fa_dh;
      s.n_seg = 4;
      s.row_begin[0] = 0; s.row_end[0] = qd; s.src[0] = static_cast<const uint8_t*>(lw.w_q);
      s.row_begin[1] = qd; s.row_end[1] = 2 * qd; s.src[1] = static_cast<const uint8_t*>(lw.w_g);
      s.row_begin[2] = 2 * qd; s.row_end[2] = 2 * qd + kd; s.src[2] = static_cast<const uint8_t*>(lw.w_k);
      s.row_begin[3] = 2 * qd + kd; s.row_end[3] = 2 * qd + 2 * kd; s.src[3] = static_cast<const uint8_t*>(lw.w_v);
    }
    ok = ok && pack(p.in[l], s);
    if (!lw.w_o || !lw.w_gate || !lw.w_up || !lw.w_down || !lw.attn_norm || !lw.ffn_norm) { ok = false; break; }
    PackSrc so{};
    so.n_seg = 1; so.row_begin[0] = 0; so.row_end[0] = H; so.src[0] = static_cast<const uint8_t*>(lw.w_o);
    ok = ok && pack(p.o[l], so);
    PackSrc sg{};
    sg.n_seg = 2; sg.interleave_gate_up = 1;
    sg.row_begin[0] = 0; sg.row_end[0] = F; sg.src[0] = static_cast<const uint8_t*>(lw.w_gate);
    sg.row_begin[1] = 0; sg.row_end[1] = F; sg.src[1] = static_cast<const uint8_t*>(lw.w_up);
    ok = ok && pack(p.gu[l], sg);
    PackSrc sd{};
    sd.n_seg = 1; sd.row_begin[0] = 0; sd.row_end[0] = H; sd.src[0] = static_cast<const uint8_t*>(lw.w_down);
    ok = ok && pack(p.down[l], sd);
    // small fp32 parameters
    ok = ok && cudaMemcpyAsync(packed + p.off_attn_norm[l], lw.attn_norm, H * 4, cudaMemcpyDeviceToDevice, c->stream) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(packed + p.off_ffn_norm[l], lw.ffn_norm, H * 4, cudaMemcpyDeviceToDevice, c->stream) == cudaSuccess;
    if (gdn) {
      ok = ok && cudaMemcpyAsync(packed + p.off_conv[l], lw.conv_w, static_cast<size_t>(p.conv_ch) * 16, cudaMemcpyDeviceToDevice, c->stream) == cudaSuccess;
      ok = ok && cudaMemcpyAsync(packed + p.off_onorm[l], lw.o_norm, L.gdn_dv * 4, cudaMemcpyDeviceToDevice, c->stream) == cudaSuccess;
    }
  }
  if (!ok) { mk_free(c); return MK_ERR_INVALID; }
  {
    PackSrc sl{};
    sl.n_seg = 1; sl.row_begin[0] = 0; sl.row_end[0] = L.vocab;
    sl.src[0] = static_cast<const uint8_t*>(L.tied_lm_head ? w->embed : w->lm_head);
    ok = pack(p.lm, sl);
    ok = ok && cudaMemcpyAsync(packed + p.off_embed, w->embed, q4_bytes(L.vocab, H), cudaMemcpyDeviceToDevice, c->stream) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(packed + p.off_final_norm, w->final_norm, H * 4, cudaMemcpyDeviceToDevice, c->stream) == cudaSuccess;
  }
  if (!ok) { mk_free(c); return MK_ERR_CUDA; }
  if (L.has_mtp) {
    const mk_layer_weights& mw = w->mtp;
    const int M = MK_MAX_LAYERS;
    if (!w->mtp_fc || !w->mtp_norm_h || !w->mtp_norm_e || !w->mtp_final_norm || !mw.w_q || !mw.w_g || !mw.w_k ||
        !mw.w_v || !mw.w_o || !mw.w_gate || !mw.w_up || !mw.w_down || !mw.attn_norm || !mw.ffn_norm) {
      mk_free(c);
      return MK_ERR_INVALID;
    }
    const int qd = L.fa_hq * L.fa_dh, kd = L.fa_hkv * L.fa_dh;
    PackSrc sf{};
    sf.n_seg = 1; sf.row_begin[0] = 0; sf.row_end[0] = H; sf.src[0] = static_cast<const uint8_t*>(w->mtp_fc);
    ok = pack(p.mtp_fc, sf);
    PackSrc s{};
    s.n_seg = 4;
    s.row_begin[0] = 0; s.row_end[0] = qd; s.src[0] = static_cast<const uint8_t*>(mw.w_q);
    s.row_begin[1] = qd; s.row_end[1] = 2 * qd; s.src[1] = static_cast<const uint8_t*>(mw.w_g);
    s.row_begin[2] = 2 * qd; s.row_end[2] = 2 * qd + kd; s.src[2] = static_cast<const uint8_t*>(mw.w_k);
    s.row_begin[3] = 2 * qd + kd; s.row_end[3] = 2 * qd + 2 * kd; s.src[3] = static_cast<const uint8_t*>(mw.w_v);
    ok = ok && pack(p.in[M], s);
    PackSrc so{};
    so.n_seg = 1; so.row_begin[0] = 0; so.row_end[0] = H; so.src[0] = static_cast<const uint8_t*>(mw.w_o);
    ok = ok && pack(p.o[M], so);
    PackSrc sg{};
    sg.n_seg = 2; sg.interleave_gate_up = 1;
    sg.row_begin[0] = 0; sg.row_end[0] = F; sg.src[0] = static_cast<const uint8_t*>(mw.w_gate);
    sg.row_begin[1] = 0; sg.row_end[1] = F; sg.src[1] = static_cast<const uint8_t*>(mw.w_up);
    ok = ok && pack(p.gu[M], sg);
    PackSrc sd{};
    sd.n_seg = 1; sd.row_begin[0] = 0; sd.row_end[0] = H; sd.src[0] = static_cast<const uint8_t*>(mw.w_down);
    ok = ok && pack(p.down[M], sd);
    auto vec = [&](size_t off, const float* src) {
      return cudaMemcpyAsync(packed + off, src, H * 4, cudaMemcpyDeviceToDevice, c->stream) == cudaSuccess;
    };
    ok = ok && vec(p.off_attn_norm[M], mw.attn_norm) && vec(p.off_ffn_norm[M], mw.ffn_norm) &&
         vec(p.off_mtp_norm_h, w->mtp_norm_h) && vec(p.off_mtp_norm_e, w->mtp_norm_e) &&
         vec(p.off_mtp_final_norm, w->mtp_final_norm);
    if (!ok) { mk_free(c); return MK_ERR_CUDA; }
  }

  // ---- launch geometry
  int bps = 0;
  if (configure_persistent(&bps) != cudaSuccess || bps < 1) { mk_free(c); return MK_ERR_LAUNCH; }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { mk_free(c); return MK_ERR_CUDA; }
  c->device = dev;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  c->grid = sms;  // one block per SM: the block owns the SM's shared memory

  // ---- descriptors and scratch
  ModelDesc& md = c->md_host;
  std::memset(&md, 0, sizeof(md));
  md.n_layers = L.n_layers; md.H = H; md.F = F; md.V = L.vocab;
  md.hq = L.fa_hq; md.hkv = L.fa_hkv; md.dh = L.fa_dh;
  md.hk = L.gdn_hk; md.hv = L.gdn_hv; md.dk = L.gdn_dk; md.dv = L.gdn_dv; md.cw = L.conv_w;
  md.conv_ch = p.conv_ch; md.n_gdn = p.n_gdn; md.n_fa = p.n_fa;
  md.n_in_max = p.n_in_max; md.o_stride = p.o_stride;
  md.kv_q8 = L.kv_dtype == MK_KV_Q8; md.page_tokens = L.page_tokens; md.n_pages = L.n_pages;
  md.max_pages_per_seq = L.max_pages_per_seq; md.n_slots = L.n_state_slots; md.max_seqs = L.max_seqs;
  md.grid = c->grid; md.eps = L.rms_eps;
  int gi = 0, fi = 0, max_tiles = 1;
  auto gemm = [&](GemmDesc& g, const PhasePlan& ph, int pro, int epi, const float* gain) {
    g.w = packed + ph.off; g.n_tiles = ph.n_tiles; g.nsb = ph.nsb; g.n_out = ph.n_out;
    g.pro = pro; g.epi = epi; g.gain = gain;
    g.zero_buf = ZERO_NONE;
    max_tiles = std::max(max_tiles, ph.n_tiles);
  };
  for (int l = 0; l < L.n_layers; ++l) {
    LayerDesc& ld = md.layer[l];
    const bool gdn = L.layer_kind[l] == MK_LAYER_GDN;
    ld.kind = L.layer_kind[l];
    ld.gdn_i = gdn ? gi++ : -1;
    ld.fa_i = gdn ? -1 : fi++;
    gemm(ld.in, p.in[l], PRO_RMS_X, EPI_STORE_YIN, reinterpret_cast<const float*>(packed + p.off_attn_norm[l]));
    gemm(ld.o, p.o[l], gdn ? PRO_GDN_OUT : PRO_FA_OUT, EPI_RESID_X,
         gdn ? reinterpret_cast<const float*>(packed + p.off_onorm[l]) : nullptr);
    gemm(ld.gu, p.gu[l], PRO_RMS_X, EPI_STORE_GU, reinterpret_cast<const float*>(packed + p.off_ffn_norm[l]));
    gemm(ld.down, p.down[l], PRO_H, EPI_RESID_X, nullptr);
    ld.conv_w = gdn ? reinterpret_cast<const float*>(packed + p.off_conv[l]) : nullptr;
  }
  gemm(md.lm, p.lm, PRO_RMS_X, EPI_TOP2, reinterpret_cast<const float*>(packed + p.off_final_norm));
  md.lm.dump = 1;
  if (L.has_mtp) {
    // the MTP block is layer n_layers: a gated-attention layer on KV layer n_fa
    const int M = MK_MAX_LAYERS;
    LayerDesc& ld = md.layer[L.n_layers];
    ld.kind = MK_LAYER_FA;
    ld.gdn_i = -1;
    ld.fa_i = fi;
    gemm(ld.in, p.in[M], PRO_RMS_X, EPI_STORE_YIN, reinterpret_cast<const float*>(packed + p.off_attn_norm[M]));
    gemm(ld.o, p.o[M], PRO_FA_OUT, EPI_RESID_X, nullptr);
    gemm(ld.gu, p.gu[M], PRO_RMS_X, EPI_STORE_GU, reinterpret_cast<const float*>(packed + p.off_ffn_norm[M]));
    gemm(ld.down, p.down[M], PRO_H, EPI_RESID_X, nullptr);
    ld.o.zero_buf = ZERO_GU;
    ld.down.zero_buf = ZERO_YIN;
    ld.conv_w = nullptr;
    gemm(md.mtp_fc, p.mtp_fc, PRO_MTP_IN, EPI_RESID_X, nullptr);
    // the draft lm_head is the first tiles of the packed lm_head (rows [0, draft_vocab))
    PhasePlan dl = p.lm;
    dl.n_tiles = tiles_of(L.draft_vocab);
    dl.n_out = L.draft_vocab;
    gemm(md.mtp_lm, dl, PRO_RMS_X, EPI_TOP2, reinterpret_cast<const float*>(packed + p.off_mtp_final_norm));
    md.has_mtp = 1;
    md.n_draft = L.n_draft;
    md.draft_vocab = L.draft_vocab;
    md.mtp_norm_h = reinterpret_cast<const float*>(packed + p.off_mtp_norm_h);
    md.mtp_norm_e = reinterpret_cast<const float*>(packed + p.off_mtp_norm_e);
  }
  // split tiles are summed into buffers that must start at zero: the
  // gate/up sums are cleared during o_proj, the next input projections during down
  for (int l = 0; l < L.n_layers; ++l) {
    md.layer[l].o.zero_buf = ZERO_GU;
    md.layer[l].down.zero_buf = ZERO_YIN;
  }
  md.final_norm = reinterpret_cast<const float*>(packed + p.off_final_norm);
  md.embed = packed + p.off_embed;
  md.kv_k = b->kv_k; md.kv_v = b->kv_v;
  md.kv_ks = static_cast<uint16_t*>(b->kv_k_scale); md.kv_vs = static_cast<uint16_t*>(b->kv_v_scale);
  const int n_kv = n_kv_of(&L);
  if (n_kv > 0 && (!encode_kv_map(&c->tm_k, b->kv_k, L, n_kv) || !encode_kv_map(&c->tm_v, b->kv_v, L, n_kv))) {
    mk_free(c);
    return MK_ERR_CUDA;
  }
  md.gdn_state = b->gdn_state; md.conv_state = b->conv_state;

  md.part_rows = std::min(kMaxQRows, kMaxT * (L.fa_hq / std::max(1, L.fa_hkv)));
  md.part_stride = std::max(1, L.fa_dh) + 4;
  const size_t nrec = static_cast<size_t>(c->grid) * kWarps;
  const size_t attn_items_max = static_cast<size_t>(2 * c->grid + kMaxSeqs * std::max(1, L.fa_hkv));
  c->tickets_bytes = static_cast<size_t>(max_tiles) * 4;
  // the attention split counters, then the RMSNorm slice counters (one per GEMM phase)
  const size_t attn_counters = static_cast<size_t>(kMaxSeqs) * std::max(1, L.fa_hkv);
  c->attn_tickets_bytes = (attn_counters + gemm_phases(L)) * 4;
  if ((dev_alloc(c, &md.x, static_cast<size_t>(kMaxRows) * H * 4)) ||
      (dev_alloc(c, &md.yin, static_cast<size_t>(kMaxRows) * p.n_in_max * 4)) ||
      (dev_alloc(c, &md.o, static_cast<size_t>(kMaxRows) * std::max(1, p.o_stride) * 4)) ||
      (dev_alloc(c, &md.h, static_cast<size_t>(kMaxRows) * F * 4)) ||
      (dev_alloc(c, &md.gu, static_cast<size_t>(kMaxRows) * 2 * F * 4)) ||
      (dev_alloc(c, &md.logits, static_cast<size_t>(kMaxRows) * L.vocab * 4)) ||
      (dev_alloc(c, &md.tickets, c->tickets_bytes)) ||
      (dev_alloc(c, &md.attn_part, attn_items_max * kMaxAttnGroups * md.part_rows * md.part_stride * 4)) ||
      (dev_alloc(c, &md.attn_tickets, c->attn_tickets_bytes)) ||
      (dev_alloc(c, &md.norm_part, static_cast<size_t>(gemm_phases(L)) * kMaxNormSlices * kMaxRows * 4)) ||
      (dev_alloc(c, &md.top_val, nrec * kMaxRows * 4)) ||
      (dev_alloc(c, &md.top_idx, nrec * kMaxRows * 4)) ||
      (dev_alloc(c, &md.page_table, static_cast<size_t>(L.max_seqs) * L.max_pages_per_seq * 4)) ||
      (dev_alloc(c, &md.out, kOutInts * 4)) ||
      (dev_alloc(c, &md.bar, 64)) ||
      (dev_alloc(c, &md.err, 64)) ||
      (dev_alloc(c, &md.mtp_in, L.has_mtp ? static_cast<size_t>(kMaxRows) * 2 * H * 4 : 0)) ||
      (dev_alloc(c, &md.mtp_h, L.has_mtp ? static_cast<size_t>(kMaxSeqs) * H * 4 : 0)) ||
      (dev_alloc(c, &md.mtp_rope, static_cast<size_t>(kMaxSeqs) * (kMaxDh / 2) * sizeof(float2))) ||
      (dev_alloc(c, &md.mtp_row, static_cast<size_t>(kMaxSeqs) * 2 * 4)) ||
      (dev_alloc(c, &c->inv_freq, (kMaxDh / 2) * sizeof(double))) ||
      (dev_alloc(c, &c->md_dev, sizeof(ModelDesc))) ||
      (dev_alloc(c, &c->sd_dev, sizeof(StepDesc)))) {
    mk_free(c);
    return MK_ERR_CUDA;
  }
  md.norm_cnt = md.attn_tickets + attn_counters;
  if (cudaMallocHost(&c->sd_host, sizeof(StepDesc)) != cudaSuccess ||
      cudaMallocHost(&c->out_host, (kOutInts + 16) * 4) != cudaSuccess ||
      cudaMallocHost(&c->pt_host, static_cast<size_t>(L.max_seqs) * L.max_pages_per_seq * 4) != cudaSuccess ||
      cudaEventCreate(&c->ev0) != cudaSuccess || cudaEventCreate(&c->ev1) != cudaSuccess) {
    mk_free(c);
    return MK_ERR_CUDA;
  }
  // RoPE inverse frequencies in double, for the angles the draft passes compute on the device
  double inv_freq[kMaxDh / 2] = {0.0};
  for (int i = 0; i < L.fa_dh / 2; ++i)
    inv_freq[i] = std::pow(static_cast<double>(L.rope_base), -2.0 * i / std::max(1, L.fa_dh));
  md.inv_freq = c->inv_freq;
  if (cudaMemcpyAsync(c->inv_freq, inv_freq, sizeof(inv_freq), cudaMemcpyHostToDevice, c->stream) != cudaSuccess ||
      cudaMemcpyAsync(c->md_dev, &md, sizeof(ModelDesc), cudaMemcpyHostToDevice, c->stream) != cudaSuccess ||
      cudaStreamSynchronize(c->stream) != cudaSuccess) {
    mk_free(c);
    return MK_ERR_CUDA;
  }
  c->seqs.resize(L.max_seqs);
  for (int i = 0; i < L.n_pages; ++i) c->free_pages.insert(i);
  *out = c;
  return MK_OK;
}

mk_status mk_seq_set(mk_ctx* c, int32_t seq, int32_t length, const int32_t* pages, int32_t n_pages) {
  if (!c || seq < 0 || seq >= c->L.max_seqs || length < 0 || n_pages < 0) return MK_ERR_INVALID;
  if (n_pages > c->L.max_pages_per_seq || (n_pages && !pages)) return MK_ERR_INVALID;
  if (n_pages * c->L.page_tokens < length) return MK_ERR_INVALID;
  SeqInfo& s = c->seqs[seq];
  std::set<int> avail = c->free_pages;
  for (int p : s.pages) avail.insert(p);
  for (int i = 0; i < n_pages; ++i) {
    if (!avail.count(pages[i])) return MK_ERR_INVALID;
    avail.erase(pages[i]);
  }
  c->free_pages = avail;
  s = SeqInfo();
  s.used = true;
  s.len = length;
  s.pages.assign(pages, pages + n_pages);
  s.slot = 0;
  if (upload_pages(c, seq) != cudaSuccess || cudaStreamSynchronize(c->stream) != cudaSuccess) return MK_ERR_CUDA;
  return MK_OK;
}

mk_status mk_seq_reset(mk_ctx* c, int32_t seq) {
  if (!c || seq < 0 || seq >= c->L.max_seqs) return MK_ERR_INVALID;
  SeqInfo& s = c->seqs[seq];
  for (int p : s.pages) c->free_pages.insert(p);
  s = SeqInfo();
  return MK_OK;
}

mk_status mk_seq_get(mk_ctx* c, int32_t seq, int32_t* length, int32_t* pages, int32_t* n_pages,
                     int32_t* state_slot) {
  if (!c || seq < 0 || seq >= c->L.max_seqs) return MK_ERR_INVALID;
  const SeqInfo& s = c->seqs[seq];
  if (length) *length = s.len;
  if (n_pages) *n_pages = static_cast<int32_t>(s.pages.size());
  if (pages) for (size_t i = 0; i < s.pages.size(); ++i) pages[i] = s.pages[i];
  if (state_slot) *state_slot = s.slot;
  return MK_OK;
}

mk_status mk_commit(mk_ctx* c, int32_t n, const int32_t* seq_ids, const int32_t* n_keep) {
  if (!c || n < 0 || (n && (!seq_ids || !n_keep))) return MK_ERR_INVALID;
  for (int i = 0; i < n; ++i) {
    if (seq_ids[i] < 0 || seq_ids[i] >= c->L.max_seqs) return MK_ERR_INVALID;
    const SeqInfo& s = c->seqs[seq_ids[i]];
    if (!s.pending) return MK_ERR_PENDING;
    if (n_keep[i] < 1 || n_keep[i] > s.count) return MK_ERR_INVALID;
  }
  for (int i = 0; i < n; ++i) commit_seq(c, c->seqs[seq_ids[i]], n_keep[i]);
  return MK_OK;
}

mk_status mk_debug_outputs(mk_ctx* c, float* logits, float* hidden) {
  if (!c) return MK_ERR_INVALID;
  c->md_host.dbg_logits = logits;
  c->md_host.dbg_hidden = hidden;
  if (cudaMemcpyAsync(c->md_dev, &c->md_host, sizeof(ModelDesc), cudaMemcpyHostToDevice, c->stream) != cudaSuccess ||
      cudaStreamSynchronize(c->stream) != cudaSuccess)
    return MK_ERR_CUDA;
  return MK_OK;
}

mk_status mk_debug_q8_encode(const float* x, int64_t n_blocks, int8_t* q, uint16_t* d16, void* stream) {
  if (n_blocks < 0 || (n_blocks > 0 && (!x || !q || !d16))) return MK_ERR_INVALID;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_q8_encode(x, n_blocks, q, d16, s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
    return MK_ERR_CUDA;
  return MK_OK;
}

mk_status mk_debug_timeline(mk_ctx* c, uint64_t* stamps) {
  if (!c) return MK_ERR_INVALID;
  c->md_host.dbg_time = stamps;
  if (cudaMemcpyAsync(c->md_dev, &c->md_host, sizeof(ModelDesc), cudaMemcpyHostToDevice, c->stream) != cudaSuccess ||
      cudaStreamSynchronize(c->stream) != cudaSuccess)
    return MK_ERR_CUDA;
  return MK_OK;
}

mk_status mk_debug_skip_arrival(mk_ctx* c, int32_t block, int32_t barrier, uint64_t timeout_ns) {
  if (!c) return MK_ERR_INVALID;
  c->skip_block = block;
  c->skip_barrier = barrier;
  c->barrier_timeout_ns = timeout_ns ? timeout_ns : 500000000ull;
  return MK_OK;
}

mk_status mk_debug_scratch(mk_ctx* c, int32_t rows, float* x, float* y, float* o, float* h,
                           int32_t* y_stride, int32_t* o_stride) {
  if (!c || rows < 0 || rows > kMaxRows) return MK_ERR_INVALID;
  const ModelDesc& md = c->md_host;
  if (y_stride) *y_stride = md.n_in_max;
  if (o_stride) *o_stride = md.o_stride;
  const size_t n = static_cast<size_t>(rows);
  if ((x && cudaMemcpyAsync(x, md.x, n * md.H * 4, cudaMemcpyDeviceToHost, c->stream)) ||
      (y && cudaMemcpyAsync(y, md.yin, n * md.n_in_max * 4, cudaMemcpyDeviceToHost, c->stream)) ||
      (o && cudaMemcpyAsync(o, md.o, n * md.o_stride * 4, cudaMemcpyDeviceToHost, c->stream)) ||
      (h && cudaMemcpyAsync(h, md.h, n * md.F * 4, cudaMemcpyDeviceToHost, c->stream)) ||
      cudaStreamSynchronize(c->stream))
    return MK_ERR_CUDA;
  return MK_OK;
}

mk_status mk_step_io_bytes(mk_ctx* c, uint64_t* h2d, uint64_t* d2h) {
  if (!c) return MK_ERR_INVALID;
  if (h2d) *h2d = c->h2d_bytes;
  if (d2h) *d2h = c->d2h_bytes;
  return MK_OK;
}

int32_t mk_grid_blocks(mk_ctx* c) { return c ? c->grid : 0; }

mk_status mk_step_prepare(mk_ctx* c, int32_t n_rows, const int32_t* tokens, const int32_t* positions,
                          const int32_t* seq_ids, const uint8_t* row_flags) {
  if (!c || n_rows < 1 || n_rows > kMaxRows || !tokens || !positions || !seq_ids) return MK_ERR_INVALID;
  const mk_layout& L = c->L;
  c->prepared = c->launched = false;
  // group rows into contiguous runs of one sequence each
  int n_seq = 0, row0[kMaxSeqs], T[kMaxSeqs], sid[kMaxSeqs], prompt[kMaxSeqs];
  for (int r = 0; r < n_rows; ++r) {
    const int f = row_flags ? row_flags[r] : 0;
    if (f > 2) return MK_ERR_INVALID;
    if (f != 0 && L.has_mtp) return MK_ERR_UNSUPPORTED;  // the MTP head runs over verified rows only
    if (tokens[r] < 0 || tokens[r] >= L.vocab) return MK_ERR_INVALID;
    const int s = seq_ids[r];
    if (s < 0 || s >= L.max_seqs || !c->seqs[s].used) return MK_ERR_INVALID;
    if (r == 0 || s != seq_ids[r - 1]) {
      for (int i = 0; i < n_seq; ++i)
        if (sid[i] == s) return MK_ERR_INVALID;
      if (n_seq == kMaxSeqs) return MK_ERR_INVALID;
      sid[n_seq] = s; row0[n_seq] = r; T[n_seq] = 0; prompt[n_seq] = f; ++n_seq;
    } else {
      // every row of a sequence is of one kind; flag 2 (ends the prompt) only on its last row
      const int prev = prompt[n_seq - 1];
      if ((f != 0) != (prev != 0) || prev == 2) return MK_ERR_INVALID;
      prompt[n_seq - 1] = f;  // the sequence's kind is its last row's flag
    }
    ++T[n_seq - 1];
  }
  const int grp = L.fa_hq / std::max(1, L.fa_hkv);
  for (int i = 0; i < n_seq; ++i) {
    if (T[i] > kMaxT || T[i] + 1 > L.n_state_slots || T[i] * grp > kMaxQRows) return MK_ERR_UNSUPPORTED;
  }
  // positions the step may write per sequence beyond its rows: the MTP draft
  // passes after the last row
  const int extra = L.has_mtp ? L.n_draft - 1 : 0;
  // positions must continue each sequence (after its pending step is kept)
  for (int i = 0; i < n_seq; ++i) {
    const SeqInfo& s = c->seqs[sid[i]];
    const int base = s.len + (s.pending ? s.count : 0);
    for (int j = 0; j < T[i]; ++j)
      if (positions[row0[i] + j] != base + j) return MK_ERR_INVALID;
    if ((base + T[i] + extra + L.page_tokens - 1) / L.page_tokens > L.max_pages_per_seq) return MK_ERR_NO_PAGES;
  }
  // page demand check before touching any state: pages a pending step does
  // not keep are released by its auto-commit first
  {
    int need = 0, released = 0;
    for (int i = 0; i < n_seq; ++i) {
      const SeqInfo& s = c->seqs[sid[i]];
      int have = static_cast<int>(s.pages.size());
      const int len_after = s.len + (s.pending ? s.count : 0);
      if (s.pending) {
        const int keep = (len_after + L.page_tokens - 1) / L.page_tokens;
        if (have > keep) { released += have - keep; have = keep; }
      }
      const int want = (len_after + T[i] + extra + L.page_tokens - 1) / L.page_tokens;
      need += std::max(0, want - have);
    }
    if (need > static_cast<int>(c->free_pages.size()) + released) return MK_ERR_NO_PAGES;
  }
  // auto-commit pending sequences of this step
  for (int i = 0; i < n_seq; ++i) {
    SeqInfo& s = c->seqs[sid[i]];
    if (s.pending) commit_seq(c, s, s.count);
  }
  // page allocation, lowest free first, in row order (a sequence's last row
  // also covers its draft passes' positions)
  for (int r = 0; r < n_rows; ++r) {
    SeqInfo& s = c->seqs[seq_ids[r]];
    const bool last = r + 1 == n_rows || seq_ids[r + 1] != seq_ids[r];
    const int need = (positions[r] + (last ? extra : 0)) / L.page_tokens + 1;
    while (static_cast<int>(s.pages.size()) < need) {
      if (c->free_pages.empty()) return MK_ERR_NO_PAGES;
      s.pages.push_back(*c->free_pages.begin());
      c->free_pages.erase(c->free_pages.begin());
    }
  }
  StepDesc& sd = *c->sd_host;
  std::memset(&sd, 0, sizeof(StepDesc));
  sd.R = n_rows;
  sd.n_seq = n_seq;
  sd.nt = (2 * n_rows + 7) / 8;
  for (int r = 0; r < n_rows; ++r) {
    sd.row_tok[r] = tokens[r];
    sd.row_pos[r] = positions[r];
  }
  // attention: 16-token chunks of the cached context cut into about one
  // item per block, at most kMaxSplits parts per (sequence, kv head)
  int total_chunks = 0, t_max = 1;
  for (int i = 0; i < n_seq; ++i) {
    total_chunks += (c->seqs[sid[i]].len + kChunk - 1) / kChunk;
    t_max = std::max(t_max, T[i]);
  }
  const int hkv = std::max(1, L.fa_hkv);
  int cps = std::max(1, (total_chunks * hkv + c->grid - 1) / c->grid);
  int max_chunks = 1;
  for (int i = 0; i < n_seq; ++i) {
    const int nc = (c->seqs[sid[i]].len + kChunk - 1) / kChunk;
    max_chunks = std::max(max_chunks, nc);
    cps = std::max(cps, (nc + kMaxSplits - 1) / kMaxSplits);
  }
  // per-sequence rounding can push the item count past the grid; grow the
  // split until every item has a block of its own
  auto n_items = [&](int cp) {
    int n = 0;
    for (int i = 0; i < n_seq; ++i)
      n += hkv * std::max(1, ((c->seqs[sid[i]].len + kChunk - 1) / kChunk + cp - 1) / cp);
    return n;
  };
  while (cps < max_chunks && n_items(cps) > c->grid) ++cps;
  int items = 0;
  for (int i = 0; i < n_seq; ++i) {
    const SeqInfo& s = c->seqs[sid[i]];
    sd.seq_id[i] = sid[i];
    sd.seq_row0[i] = row0[i];
    sd.seq_T[i] = T[i];
    sd.seq_len[i] = s.len;
    sd.seq_slot_in[i] = s.slot;
    // verify rows keep the state after every row (the commit picks one); prompt
    // rows are committed through their last row, so only that state is written
    sd.seq_snap_all[i] = prompt[i] ? 0 : 1;
    sd.seq_prompt[i] = prompt[i];
    c->step_prompt[i] = prompt[i];
    int at = 0;
    for (int t = 0; t < T[i]; ++t) {
      if (at == s.slot) ++at;
      sd.seq_slot_out[i][t] = at;
      c->step_snap[i][t] = at;
      ++at;
    }
    const int nchunk = (s.len + kChunk - 1) / kChunk;
    sd.seq_chunks_per_split[i] = cps;
    sd.seq_nsplit[i] = std::max(1, (nchunk + cps - 1) / cps);
    sd.seq_item0[i] = items;
    items += hkv * sd.seq_nsplit[i];
    for (int j = 0; j < T[i]; ++j) sd.row_si[row0[i] + j] = i;
    c->step_seq[i] = sid[i];
    c->step_T[i] = T[i];
  }
  sd.n_attn_items = items;
  // the splits of one (sequence, kv head) wait for each other before merging:
  // every item needs a block of its own; an item's page ids fit the block's page list
  if (items > c->grid || cps > kAttnPageList) return MK_ERR_UNSUPPORTED;
  if (L.fa_dh > 0) {
    attn_plan(t_max * (L.fa_hq / hkv), L.fa_dh, L.kv_dtype == MK_KV_Q8, kRingBytes, sd.attn_nq, sd.attn_jw,
              sd.attn_wpg, sd.attn_ng, sd.attn_spg, sd.attn_nslots);
    if (sd.attn_spg < 1) return MK_ERR_UNSUPPORTED;
    // the merge's weights of every (sequence, kv head) fit below the phase's flag word
    for (int i = 0; i < n_seq; ++i) {
      const int qrows = T[i] * (L.fa_hq / hkv), parts = sd.seq_nsplit[i] * sd.attn_ng;
      if (2 * qrows * parts + qrows > kAttnCombineFloats) return MK_ERR_UNSUPPORTED;
    }
  }
  sd.skip_block = c->skip_block;
  sd.skip_barrier = c->skip_barrier;
  sd.barrier_timeout_ns = c->barrier_timeout_ns;
  if (L.fa_dh > 0) {
    for (int r = 0; r < n_rows; ++r)
      for (int i = 0; i < L.fa_dh / 2; ++i) {
        const double theta = static_cast<double>(positions[r]) *
                             std::pow(static_cast<double>(L.rope_base), -2.0 * i / L.fa_dh);
        sd.rope[r][i] = make_float2(static_cast<float>(std::cos(theta)), static_cast<float>(std::sin(theta)));
      }
  }
  c->n_rows = n_rows;
  c->n_seq = n_seq;
  c->h2d_bytes = sizeof(StepDesc);
  for (int i = 0; i < n_seq; ++i)
    if (upload_pages(c, sid[i]) != cudaSuccess) return MK_ERR_CUDA;
  if (cudaMemcpyAsync(c->sd_dev, c->sd_host, sizeof(StepDesc), cudaMemcpyHostToDevice, c->stream) != cudaSuccess)
    return MK_ERR_CUDA;
  c->prepared = true;
  return MK_OK;
}

mk_status mk_step_launch(mk_ctx* c) {
  if (!c || !c->prepared) return MK_ERR_INVALID;
  // the barrier counter and the attention split counters count up within one launch
  if (cudaMemsetAsync(c->md_host.bar, 0, 64, c->stream) != cudaSuccess ||
      cudaMemsetAsync(c->md_host.err, 0, 64, c->stream) != cudaSuccess ||
      cudaMemsetAsync(c->md_host.attn_tickets, 0, c->attn_tickets_bytes, c->stream) != cudaSuccess)
    return MK_ERR_CUDA;
  cudaEventRecord(c->ev0, c->stream);
  const cudaError_t e =
      launch_persistent(c->md_dev, c->sd_dev, c->grid, &c->tm_k, &c->tm_v, c->stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e == cudaErrorCooperativeLaunchTooLarge ? MK_ERR_LAUNCH : MK_ERR_CUDA;
  }
  cudaEventRecord(c->ev1, c->stream);
  c->launched = true;
  c->timed = true;
  return MK_OK;
}

mk_status mk_step_finish(mk_ctx* c, int32_t* out_tokens, int32_t* out_counts) {
  if (!c || !c->launched) return MK_ERR_INVALID;
  c->drafts.clear();
  int32_t* h = c->out_host;
  if (cudaMemcpyAsync(h, c->md_host.out, kOutInts * 4, cudaMemcpyDeviceToHost, c->stream) != cudaSuccess ||
      cudaMemcpyAsync(h + kOutInts, c->md_host.err, 16, cudaMemcpyDeviceToHost, c->stream) != cudaSuccess ||
      cudaStreamSynchronize(c->stream) != cudaSuccess) {
    c->prepared = c->launched = false;
    return MK_ERR_CUDA;
  }
  c->prepared = c->launched = false;
  c->d2h_bytes = kOutInts * 4 + 16;
  const int32_t dev_err = h[kOutInts], nonfinite = h[kOutInts + 1];
  if (dev_err != DEV_OK) {
    cudaMemsetAsync(c->md_host.tickets, 0, c->tickets_bytes, c->stream);
    cudaMemsetAsync(c->md_host.attn_tickets, 0, c->attn_tickets_bytes, c->stream);
    cudaStreamSynchronize(c->stream);
    return MK_ERR_BARRIER_TIMEOUT;
  }
  if (c->L.has_mtp)
    for (int i = 0; i < c->n_seq; ++i)
      for (int j = 0; j < c->L.n_draft; ++j) c->drafts.push_back(h[kOutDrafts + i * kMaxDraft + j]);
  if (!finish_seqs(c, h, out_tokens, out_counts)) return MK_ERR_CUDA;
  return nonfinite ? MK_ERR_NONFINITE : MK_OK;
}

mk_status mk_step(mk_ctx* c, int32_t n_rows, const int32_t* tokens, const int32_t* positions,
                  const int32_t* seq_ids, const uint8_t* row_flags, int32_t* out_tokens, int32_t* out_counts) {
  mk_status s = mk_step_prepare(c, n_rows, tokens, positions, seq_ids, row_flags);
  if (s != MK_OK) return s;
  s = mk_step_launch(c);
  if (s != MK_OK) return s;
  return mk_step_finish(c, out_tokens, out_counts);
}

mk_status mk_last_drafts(mk_ctx* c, int32_t* drafts) {
  if (!c || !drafts || !c->L.has_mtp || c->drafts.empty()) return MK_ERR_INVALID;
  std::copy(c->drafts.begin(), c->drafts.end(), drafts);
  return MK_OK;
}

float mk_last_launch_ms(mk_ctx* c) {
  if (!c || !c->timed) return -1.f;
  float ms = -1.f;
  if (cudaEventElapsedTime(&ms, c->ev0, c->ev1) != cudaSuccess) return -1.f;
  return ms;
}

}  // extern "C"

// ------------------------------------------------------------------------
// Allocation-free step. Everything the persistent kernel writes as per-step
// scratch (residual and activation rows, split-K partials and their tickets,
// attention partials and tickets, per-warp argmax records, the result block,
// the barrier and error words, the staging rows of the attention phase, and
// the kernel's copy of the model descriptor that points at them) lives in the
// file-scope array below instead of buffers from cudaMalloc. It is sized once
// for the life of the process and shared by every call on the same device.
namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB per device
__device__ __align__(256) unsigned char g_mk_static_scratch[kStaticScratchBytes];
constexpr int kMaxDevices = 64;
void* g_static_addr[kMaxDevices] = {nullptr};

struct StaticLayout {
  size_t md, x, yin, o, h, gu, logits, tickets, attn_part, attn_tickets, norm_part, top_val, top_idx, out, bar, err,
      total;
};

StaticLayout static_layout(const mk_ctx* c, int n_attn_items) {
  const ModelDesc& md = c->md_host;
  const size_t nrec = static_cast<size_t>(c->grid) * kWarps;
  StaticLayout L{};
  size_t at = 0;
  auto take = [&](size_t& off, size_t bytes) { off = at; at = align_up(at + (bytes ? bytes : 16)); };
  take(L.md, sizeof(ModelDesc));
  take(L.x, static_cast<size_t>(kMaxRows) * md.H * 4);
  take(L.yin, static_cast<size_t>(kMaxRows) * md.n_in_max * 4);
  take(L.o, static_cast<size_t>(kMaxRows) * std::max(1, md.o_stride) * 4);
  take(L.h, static_cast<size_t>(kMaxRows) * md.F * 4);
  take(L.gu, static_cast<size_t>(kMaxRows) * 2 * md.F * 4);
  take(L.logits, static_cast<size_t>(kMaxRows) * md.V * 4);
  take(L.tickets, c->tickets_bytes);
  take(L.attn_part, static_cast<size_t>(std::max(1, n_attn_items)) * kMaxAttnGroups * md.part_rows * md.part_stride * 4);
  take(L.attn_tickets, c->attn_tickets_bytes);
  take(L.norm_part, static_cast<size_t>(gemm_phases(c->L)) * kMaxNormSlices * kMaxRows * 4);
  take(L.top_val, nrec * kMaxRows * 4);
  take(L.top_idx, nrec * kMaxRows * 4);
  take(L.out, kOutInts * 4);
  take(L.bar, 64);
  take(L.err, 64);
  L.total = at;
  return L;
}

}  // namespace

extern "C" mk_status mk_step_static(mk_ctx* c, int32_t n_rows, const int32_t* tokens, const int32_t* positions,
                                    const int32_t* seq_ids, const uint8_t* row_flags, int32_t* out_tokens,
                                    int32_t* out_counts) {
  if (!c) return MK_ERR_INVALID;
  if (c->L.has_mtp) return MK_ERR_UNSUPPORTED;
  // The worst case of this context (every attention item a step can have)
  // must fit, so that the check happens before any bookkeeping changes.
  const int worst_items = c->grid + kMaxSeqs * std::max(1, c->L.fa_hkv);
  if (static_layout(c, worst_items).total > kStaticScratchBytes) return MK_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MK_ERR_CUDA;
  // the array's address is per device: the context's device must be current
  if (dev != c->device) return MK_ERR_INVALID;
  if (!g_static_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_mk_static_scratch) != cudaSuccess || !p) return MK_ERR_CUDA;
    g_static_addr[dev] = p;
  }
  mk_status st = mk_step_prepare(c, n_rows, tokens, positions, seq_ids, row_flags);
  if (st != MK_OK) return st;
  c->prepared = false;
  const StaticLayout SL = static_layout(c, c->sd_host->n_attn_items);
  uint8_t* base = static_cast<uint8_t*>(g_static_addr[dev]);
  ModelDesc md = c->md_host;
  md.x = reinterpret_cast<float*>(base + SL.x);
  md.yin = reinterpret_cast<float*>(base + SL.yin);
  md.o = reinterpret_cast<float*>(base + SL.o);
  md.h = reinterpret_cast<float*>(base + SL.h);
  md.gu = reinterpret_cast<float*>(base + SL.gu);
  md.logits = reinterpret_cast<float*>(base + SL.logits);
  md.tickets = reinterpret_cast<uint32_t*>(base + SL.tickets);
  md.attn_part = reinterpret_cast<float*>(base + SL.attn_part);
  md.attn_tickets = reinterpret_cast<uint32_t*>(base + SL.attn_tickets);
  md.norm_cnt = md.attn_tickets + (c->md_host.norm_cnt - c->md_host.attn_tickets);
  md.norm_part = reinterpret_cast<float*>(base + SL.norm_part);
  md.top_val = reinterpret_cast<float*>(base + SL.top_val);
  md.top_idx = reinterpret_cast<int32_t*>(base + SL.top_idx);
  md.out = reinterpret_cast<int32_t*>(base + SL.out);
  md.bar = reinterpret_cast<uint32_t*>(base + SL.bar);
  md.err = reinterpret_cast<int32_t*>(base + SL.err);
  ModelDesc* md_dev = reinterpret_cast<ModelDesc*>(base + SL.md);
  // The array keeps the previous call's contents: clear what must start at zero.
  if (cudaMemcpyAsync(md_dev, &md, sizeof(ModelDesc), cudaMemcpyHostToDevice, c->stream) != cudaSuccess ||
      cudaMemsetAsync(md.tickets, 0, c->tickets_bytes, c->stream) != cudaSuccess ||
      cudaMemsetAsync(md.attn_tickets, 0, c->attn_tickets_bytes, c->stream) != cudaSuccess ||
      cudaMemsetAsync(md.bar, 0, 64, c->stream) != cudaSuccess ||
      cudaMemsetAsync(md.err, 0, 64, c->stream) != cudaSuccess ||
      cudaStreamSynchronize(c->stream) != cudaSuccess)
    return MK_ERR_CUDA;
  c->h2d_bytes += sizeof(ModelDesc);
  cudaEventRecord(c->ev0, c->stream);
  const cudaError_t e = launch_persistent(md_dev, c->sd_dev, c->grid, &c->tm_k, &c->tm_v, c->stream);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e == cudaErrorCooperativeLaunchTooLarge ? MK_ERR_LAUNCH : MK_ERR_CUDA;
  }
  cudaEventRecord(c->ev1, c->stream);
  c->timed = true;
  c->d2h_bytes = kOutInts * 4 + 16;
  int32_t* h = c->out_host;
  if (cudaMemcpyAsync(h, md.out, kOutInts * 4, cudaMemcpyDeviceToHost, c->stream) != cudaSuccess ||
      cudaMemcpyAsync(h + kOutInts, md.err, 16, cudaMemcpyDeviceToHost, c->stream) != cudaSuccess ||
      cudaStreamSynchronize(c->stream) != cudaSuccess)
    return MK_ERR_CUDA;
  if (h[kOutInts] != DEV_OK) return MK_ERR_BARRIER_TIMEOUT;
  if (!finish_seqs(c, h, out_tokens, out_counts)) return MK_ERR_CUDA;
  return h[kOutInts + 1] ? MK_ERR_NONFINITE : MK_OK;
}

extern "C" int32_t mk_debug_gemm_schedule(int32_t n_tiles, int32_t nsb, int32_t rows, int32_t grid,
                                          int32_t* warp_info, int32_t* tile_arrivals_out) {
  if (n_tiles < 1 || nsb < 1 || rows < 1 || rows > kMaxRows || grid < 1 || !warp_info || !tile_arrivals_out)
    return MK_ERR_INVALID;
  for (int cta = 0; cta < grid; ++cta)
    for (int w = 0; w < kWarps; ++w) {
      const Assign a = assign_units(n_tiles, nsb, rows, grid, cta, w);
      int32_t* o = warp_info + (static_cast<size_t>(cta) * kWarps + w) * 4;
      o[0] = a.sb0;
      o[1] = a.nsb_s;
      o[2] = static_cast<int32_t>(a.u0);
      o[3] = static_cast<int32_t>(a.u1);
    }
  const Sched sc = make_sched(nsb, rows);
  for (int t = 0; t < n_tiles; ++t)
    tile_arrivals_out[t] = static_cast<int32_t>(tile_arrivals(sc, n_tiles, nsb, grid, static_cast<uint32_t>(t)));
  return kWarps;
}

extern "C" int32_t mk_debug_act_bytes(int32_t nsb_slice, int32_t rows) { return act_bytes(nsb_slice, rows); }

extern "C" mk_status mk_debug_attn_plan(int32_t q_rows_max, int32_t dh, int32_t q8, int32_t* out) {
  if (q_rows_max < 1 || q_rows_max > kMaxQRows || dh < 64 || dh > kMaxDh || dh % 64 || !out) return MK_ERR_INVALID;
  int32_t nq, jw, wpg, ng, spg, nslots;
  attn_plan(q_rows_max, dh, q8 ? 1 : 0, kRingBytes, nq, jw, wpg, ng, spg, nslots);
  out[0] = nq;
  out[1] = jw;
  out[2] = wpg;
  out[3] = ng;
  out[4] = spg;
  out[5] = nslots;
  out[6] = attn_xoff(nq, dh, q8 ? 1 : 0);
  out[7] = attn_xslab(wpg, nq, q8 ? 1 : 0);
  out[8] = kPhaseBytes;
  out[9] = attn_slot_layout(dh, q8 ? 1 : 0).bytes;
  out[10] = kRingBytes;
  out[11] = kAttnPageListBytes;
  return spg < 1 ? MK_ERR_UNSUPPORTED : MK_OK;
}
