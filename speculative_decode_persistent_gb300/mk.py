"""Thin ctypes binding of libmk.so (include/mk.h).

Argument marshalling only: every step of the verify cycle runs in the CUDA
library. PyTorch provides device memory and the stream. Importing this module
raises if the compiled library is missing; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("MK_LIBRARY", os.path.join(_HERE, "libmk.so"))

MK_MAX_LAYERS = 64
MK_MAX_SEQS = 8
MK_MAX_DECODE_ROWS = 12
MK_MAX_T = 8
MK_LAYER_GDN, MK_LAYER_FA = 0, 1
MK_KV_F16, MK_KV_Q8 = 0, 1

STATUS = {0: "MK_OK", -1: "MK_ERR_INVALID", -2: "MK_ERR_NO_PAGES", -3: "MK_ERR_LAUNCH",
          -4: "MK_ERR_BARRIER_TIMEOUT", -5: "MK_ERR_PENDING", -6: "MK_ERR_NONFINITE",
          -7: "MK_ERR_CUDA", -8: "MK_ERR_UNSUPPORTED"}

i32, f32, vp, sz, u64 = ctypes.c_int32, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint64


class MkError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


class mk_layout(ctypes.Structure):
    _fields_ = [
        ("n_layers", i32), ("hidden", i32), ("ffn", i32), ("vocab", i32),
        ("layer_kind", i32 * MK_MAX_LAYERS),
        ("fa_hq", i32), ("fa_hkv", i32), ("fa_dh", i32), ("rope_base", f32),
        ("gdn_hk", i32), ("gdn_hv", i32), ("gdn_dk", i32), ("gdn_dv", i32), ("conv_w", i32),
        ("tied_lm_head", i32), ("has_mtp", i32), ("draft_vocab", i32),
        ("kv_dtype", i32), ("page_tokens", i32), ("n_pages", i32), ("max_seqs", i32),
        ("max_pages_per_seq", i32), ("n_state_slots", i32), ("rms_eps", f32),
        ("n_draft", i32),
    ]


LAYER_FIELDS = ["attn_norm", "w_qkv", "w_z", "w_a", "w_b", "conv_w", "o_norm", "w_q", "w_g", "w_k", "w_v",
                "w_o", "ffn_norm", "w_gate", "w_up", "w_down"]


class mk_layer_weights(ctypes.Structure):
    _fields_ = [(n, vp) for n in LAYER_FIELDS]


class mk_weights(ctypes.Structure):
    _fields_ = [("embed", vp), ("final_norm", vp), ("lm_head", vp),
                ("layers", mk_layer_weights * MK_MAX_LAYERS),
                ("mtp", mk_layer_weights), ("mtp_fc", vp), ("mtp_norm_h", vp), ("mtp_norm_e", vp),
                ("mtp_final_norm", vp)]


class mk_buffers(ctypes.Structure):
    _fields_ = [("packed", vp), ("kv_k", vp), ("kv_v", vp), ("kv_k_scale", vp), ("kv_v_scale", vp),
                ("gdn_state", vp), ("conv_state", vp)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: run __graft_entry__.build() first")
    L = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER
    sig = {
        "mk_packed_bytes": (sz, [P(mk_layout)]),
        "mk_kv_bytes": (sz, [P(mk_layout)]),
        "mk_kv_scale_bytes": (sz, [P(mk_layout)]),
        "mk_gdn_state_bytes": (sz, [P(mk_layout)]),
        "mk_conv_state_bytes": (sz, [P(mk_layout)]),
        "mk_create": (i32, [P(mk_layout), P(mk_weights), P(mk_buffers), vp, P(vp)]),
        "mk_free": (None, [vp]),
        "mk_seq_set": (i32, [vp, i32, i32, vp, i32]),
        "mk_seq_reset": (i32, [vp, i32]),
        "mk_seq_get": (i32, [vp, i32, vp, vp, vp, vp]),
        "mk_step": (i32, [vp, i32, vp, vp, vp, vp, vp, vp]),
        "mk_step_prepare": (i32, [vp, i32, vp, vp, vp, vp]),
        "mk_step_launch": (i32, [vp]),
        "mk_step_finish": (i32, [vp, vp, vp]),
        "mk_last_drafts": (i32, [vp, vp]),
        "mk_commit": (i32, [vp, i32, vp, vp]),
        "mk_debug_outputs": (i32, [vp, vp, vp]),
        "mk_last_launch_ms": (f32, [vp]),
        "mk_debug_skip_arrival": (i32, [vp, i32, i32, u64]),
        "mk_grid_blocks": (i32, [vp]),
        "mk_debug_scratch": (i32, [vp, i32, vp, vp, vp, vp, P(i32), P(i32)]),
        "mk_step_io_bytes": (i32, [vp, P(u64), P(u64)]),
        "mk_step_static": (i32, [vp, i32, vp, vp, vp, vp, vp, vp]),
        "mk_debug_timeline": (i32, [vp, vp]),
        "mk_debug_gemm_schedule": (i32, [i32, i32, i32, i32, vp, vp]),
        "mk_debug_act_bytes": (i32, [i32, i32]),
        "mk_debug_q8_encode": (i32, [vp, ctypes.c_int64, vp, vp, vp]),
        "mk_debug_attn_plan": (i32, [i32, i32, i32, vp]),
        "mk_status_str": (ctypes.c_char_p, [i32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


lib = _load()

EXPORTS = ["mk_packed_bytes", "mk_kv_bytes", "mk_kv_scale_bytes", "mk_gdn_state_bytes",
           "mk_conv_state_bytes", "mk_create", "mk_free", "mk_seq_set", "mk_seq_reset", "mk_seq_get",
           "mk_step", "mk_step_prepare", "mk_step_launch", "mk_step_finish", "mk_last_drafts", "mk_commit",
           "mk_debug_outputs", "mk_last_launch_ms", "mk_debug_skip_arrival", "mk_grid_blocks",
           "mk_status_str", "mk_debug_scratch", "mk_step_io_bytes", "mk_step_static",
           "mk_debug_timeline", "mk_debug_gemm_schedule", "mk_debug_act_bytes", "mk_debug_q8_encode",
           "mk_debug_attn_plan"]


def gemm_schedule(n_tiles: int, nsb: int, rows: int, grid: int):
    """Host-only test hook: the kernel's split of one GEMM phase.
    Returns (warp_info [grid*warps][4]: sb0, nsb_slice, u0, u1; tile_arrivals [n_tiles])."""
    import numpy as np
    info = np.zeros((grid * 16, 4), np.int32)  # room for up to 16 math warps per block
    arr = np.zeros(n_tiles, np.int32)
    nw = lib.mk_debug_gemm_schedule(n_tiles, nsb, rows, grid, info.ctypes.data, arr.ctypes.data)
    if nw < 0:
        raise MkError(nw, "mk_debug_gemm_schedule")
    return info[: grid * nw].reshape(grid, nw, 4), arr


def _np_ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(vp)


def _check(rc: int, what: str):
    if rc != 0:
        raise MkError(rc, what)


def make_layout(model: dict, kv_q8: int, n_pages: int, max_seqs: int = MK_MAX_SEQS,
                max_pages_per_seq: int | None = None, n_state_slots: int = MK_MAX_T + 1,
                n_draft: int = 0) -> mk_layout:
    """mk_layout from a model description dict (keys as in gen/configs.py);
    n_draft: drafts per step of the MTP head (models with has_mtp)."""
    L = mk_layout()
    L.n_layers, L.hidden, L.ffn, L.vocab = model["n_layers"], model["hidden"], model["ffn"], model["vocab"]
    for i, k in enumerate(model["kinds"]):
        L.layer_kind[i] = k
    L.fa_hq, L.fa_hkv, L.fa_dh, L.rope_base = model["hq"], model["hkv"], model["dh"], model["rope_base"]
    L.gdn_hk, L.gdn_hv, L.gdn_dk, L.gdn_dv, L.conv_w = (model["hk"], model["hv"], model["dk"], model["dv"],
                                                         model["conv_w"])
    L.tied_lm_head = model["tied"]
    L.has_mtp = int(model.get("has_mtp", 0))
    L.draft_vocab = int(model.get("draft_vocab", 0)) if L.has_mtp else 0
    L.n_draft = int(n_draft) if L.has_mtp else 0
    L.kv_dtype = MK_KV_Q8 if kv_q8 else MK_KV_F16
    L.page_tokens = 16
    L.n_pages = n_pages
    L.max_seqs = max_seqs
    L.max_pages_per_seq = max_pages_per_seq or n_pages
    L.n_state_slots = n_state_slots
    L.rms_eps = model["eps"]
    return L


class Engine:
    """One mk context with its device buffers (torch CUDA tensors).

    weights: canonical numpy arrays keyed like gen.configs.tensor_inventory.
    """

    def __init__(self, model: dict, weights: dict, kv_q8: int, n_pages: int, max_seqs: int = MK_MAX_SEQS,
                 device: str = "cuda:0", stream=None, max_pages_per_seq: int | None = None,
                 n_state_slots: int = MK_MAX_T + 1, n_draft: int = 0):
        import torch
        if kv_q8 and model["dh"] % 128 and model["dh"] != 64:
            # the q8 page reader assumes one 64-byte box per K/V row when rows are
            # not a multiple of 128 bytes: a q8 head dim of 192 is not supported
            raise MkError(-8, "Engine (q8 KV needs a head dim of 64 or a multiple of 128)")
        self.torch = torch
        self.model = model
        self.device = torch.device(device)
        self.layout = make_layout(model, kv_q8, n_pages, max_seqs, max_pages_per_seq, n_state_slots, n_draft)
        Lp = ctypes.byref(self.layout)
        nbytes = lib.mk_packed_bytes(Lp)
        if nbytes == 0:
            raise MkError(-8, "mk_packed_bytes (layout rejected)")
        self.stream = stream or torch.cuda.current_stream(self.device)
        u8 = torch.uint8
        self.packed = torch.empty(nbytes, dtype=u8, device=self.device)
        self.kv_k = torch.zeros(max(lib.mk_kv_bytes(Lp), 16), dtype=u8, device=self.device)
        self.kv_v = torch.zeros(max(lib.mk_kv_bytes(Lp), 16), dtype=u8, device=self.device)
        ns = lib.mk_kv_scale_bytes(Lp)
        self.kv_ks = torch.zeros(max(ns, 16), dtype=u8, device=self.device)
        self.kv_vs = torch.zeros(max(ns, 16), dtype=u8, device=self.device)
        self.gdn_state = torch.zeros(max(lib.mk_gdn_state_bytes(Lp) // 4, 4), dtype=torch.float32,
                                     device=self.device)
        self.conv_state = torch.zeros(max(lib.mk_conv_state_bytes(Lp) // 4, 4), dtype=torch.float32,
                                      device=self.device)
        # canonical weights on the device for the repack, freed afterwards
        dev = {k: torch.from_numpy(np.ascontiguousarray(v)).to(self.device) for k, v in weights.items()}
        W = mk_weights()
        W.embed = dev["embed"].data_ptr()
        W.final_norm = dev["final_norm"].data_ptr()
        W.lm_head = dev["lm_head"].data_ptr() if "lm_head" in dev else None
        for li in range(model["n_layers"]):
            for n in LAYER_FIELDS:
                key = f"layers.{li}.{n}"
                if key in dev:
                    setattr(W.layers[li], n, dev[key].data_ptr())
        if self.layout.has_mtp:
            for n in LAYER_FIELDS:
                key = f"mtp.block.{n}"
                if key in dev:
                    setattr(W.mtp, n, dev[key].data_ptr())
            W.mtp_fc = dev["mtp.fc"].data_ptr()
            W.mtp_norm_h = dev["mtp.norm_h"].data_ptr()
            W.mtp_norm_e = dev["mtp.norm_e"].data_ptr()
            W.mtp_final_norm = dev["mtp.final_norm"].data_ptr()
        B = mk_buffers()
        B.packed = self.packed.data_ptr()
        B.kv_k, B.kv_v = self.kv_k.data_ptr(), self.kv_v.data_ptr()
        B.kv_k_scale, B.kv_v_scale = self.kv_ks.data_ptr(), self.kv_vs.data_ptr()
        B.gdn_state, B.conv_state = self.gdn_state.data_ptr(), self.conv_state.data_ptr()
        ctx = vp()
        torch.cuda.synchronize(self.device)
        rc = lib.mk_create(Lp, ctypes.byref(W), ctypes.byref(B), ctypes.c_void_p(self.stream.cuda_stream),
                           ctypes.byref(ctx))
        _check(rc, "mk_create")
        self.ctx = ctx
        torch.cuda.synchronize(self.device)
        del dev
        self.max_seqs = max_seqs
        self.n_slots = n_state_slots
        self.n_gdn = sum(1 for k in model["kinds"] if k == 0)
        self.conv_ch = 2 * model["hk"] * model["dk"] + model["hv"] * model["dv"]

    # ---------------------------------------------------------------- state
    def state_views(self):
        m = self.model
        if self.n_gdn == 0:
            return None, None
        S = self.gdn_state.view(self.max_seqs, self.n_slots, self.n_gdn, m["hv"], m["dv"], m["dk"])
        C = self.conv_state.view(self.max_seqs, self.n_slots, self.n_gdn, m["conv_w"] - 1, self.conv_ch)
        return S, C

    def kv_views(self):
        m, torch = self.model, self.torch
        n_kv = sum(1 for k in m["kinds"] if k == 1) + (1 if self.layout.has_mtp else 0)
        shape = (n_kv, self.layout.n_pages, m["hkv"], 16, m["dh"])
        n = int(np.prod(shape))
        if self.layout.kv_dtype == MK_KV_Q8:
            sshape = shape[:-1] + (m["dh"] // 32,)
            ns = int(np.prod(sshape)) * 2
            return dict(kq=self.kv_k[:n].view(torch.int8).view(shape), vq=self.kv_v[:n].view(torch.int8).view(shape),
                        ks=self.kv_ks[:ns].view(torch.int16).view(sshape),
                        vs=self.kv_vs[:ns].view(torch.int16).view(sshape))
        return dict(k=self.kv_k[:2 * n].view(torch.int16).view(shape),
                    v=self.kv_v[:2 * n].view(torch.int16).view(shape))

    def load_pool(self, pool: dict):
        """Copy a canonical numpy pool (gen.synth.make_pool layout) to the device."""
        views = self.kv_views()
        for name, arr in pool.items():
            views[name].copy_(self.torch.from_numpy(np.ascontiguousarray(arr).view(
                np.int8 if arr.dtype == np.int8 else np.int16)))

    def seq_set(self, seq: int, length: int, pages, S=None, conv=None):
        """Install a sequence; S/conv (numpy fp32) go into its state slot 0."""
        Sv, Cv = self.state_views()
        if Sv is None:
            S = conv = None
        if S is not None:
            Sv[seq, 0].copy_(self.torch.from_numpy(np.ascontiguousarray(S, np.float32)))
        if conv is not None:
            Cv[seq, 0].copy_(self.torch.from_numpy(np.ascontiguousarray(conv, np.float32)))
        self.torch.cuda.synchronize(self.device)
        pages = np.ascontiguousarray(pages, np.int32)
        _check(lib.mk_seq_set(self.ctx, seq, length, _np_ptr(pages), len(pages)), "mk_seq_set")

    def seq_get(self, seq: int):
        n = self.layout.max_pages_per_seq
        length, npg, slot = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        pages = np.zeros(n, np.int32)
        _check(lib.mk_seq_get(self.ctx, seq, ctypes.byref(length), _np_ptr(pages), ctypes.byref(npg),
                              ctypes.byref(slot)), "mk_seq_get")
        Sv, Cv = self.state_views()
        return dict(length=length.value, pages=pages[: npg.value].copy(), slot=slot.value,
                    S=None if Sv is None else Sv[seq, slot.value], conv=None if Cv is None else Cv[seq, slot.value])

    def seq_reset(self, seq: int):
        _check(lib.mk_seq_reset(self.ctx, seq), "mk_seq_reset")

    def seq_new(self, seq: int):
        """Install an empty sequence (no cached token) with a zero recurrent state."""
        Sv, Cv = self.state_views()
        if Sv is not None:
            Sv[seq, 0].zero_()
            Cv[seq, 0].zero_()
            self.torch.cuda.synchronize(self.device)
        _check(lib.mk_seq_set(self.ctx, seq, 0, None, 0), "mk_seq_set")

    def clone_sequence(self, src: int, dst: int):
        """Install sequence dst as a copy of src's committed state: the same
        length, src's KV pages copied to the lowest free page ids, and src's
        committed recurrent state copied to dst's state slot 0 (device copies;
        src must have no pending step)."""
        torch = self.torch
        info = self.seq_get(src)
        used = set()
        for s in range(self.max_seqs):
            if s != dst:
                used.update(int(p) for p in self.seq_get(s)["pages"])
        free = [p for p in range(self.layout.n_pages) if p not in used]
        n = len(info["pages"])
        if len(free) < n:
            raise MkError(-3, "clone_sequence (no free pages)")
        new = np.array(free[:n], np.int32)
        if n:
            si = torch.as_tensor(info["pages"].astype(np.int64), device=self.device)
            di = torch.as_tensor(new.astype(np.int64), device=self.device)
            for v in self.kv_views().values():  # [kv layers][pages][...]
                v[:, di] = v[:, si]
        Sv, Cv = self.state_views()
        if Sv is not None:
            Sv[dst, 0].copy_(Sv[src, info["slot"]])
            Cv[dst, 0].copy_(Cv[src, info["slot"]])
        torch.cuda.synchronize(self.device)
        _check(lib.mk_seq_set(self.ctx, dst, info["length"], _np_ptr(new), n), "mk_seq_set")

    # ----------------------------------------------------------------- step
    @staticmethod
    def _rows(tokens, positions, seq_ids, flags):
        t = np.ascontiguousarray(tokens, np.int32)
        p = np.ascontiguousarray(positions, np.int32)
        s = np.ascontiguousarray(seq_ids, np.int32)
        f = None if flags is None else np.ascontiguousarray(flags, np.uint8)
        return t, p, s, f

    def step(self, tokens, positions, seq_ids, flags=None):
        t, p, s, f = self._rows(tokens, positions, seq_ids, flags)
        nseq = len({int(x) for x in s})
        out_t = np.zeros(len(t), np.int32)
        out_c = np.zeros(nseq, np.int32)
        _check(lib.mk_step(self.ctx, len(t), _np_ptr(t), _np_ptr(p), _np_ptr(s), _np_ptr(f), _np_ptr(out_t),
                           _np_ptr(out_c)), "mk_step")
        return out_t[: int(out_c.sum())], out_c

    def step_static(self, tokens, positions, seq_ids, flags=None):
        """mk_step_static: the same step with no device allocation."""
        t, p, s, f = self._rows(tokens, positions, seq_ids, flags)
        nseq = len({int(x) for x in s})
        out_t = np.zeros(len(t), np.int32)
        out_c = np.zeros(nseq, np.int32)
        _check(lib.mk_step_static(self.ctx, len(t), _np_ptr(t), _np_ptr(p), _np_ptr(s), _np_ptr(f),
                                  _np_ptr(out_t), _np_ptr(out_c)), "mk_step_static")
        return out_t[: int(out_c.sum())], out_c

    def prepare(self, tokens, positions, seq_ids, flags=None):
        t, p, s, f = self._rows(tokens, positions, seq_ids, flags)
        self._nseq = len({int(x) for x in s})
        self._nrows = len(t)
        _check(lib.mk_step_prepare(self.ctx, len(t), _np_ptr(t), _np_ptr(p), _np_ptr(s), _np_ptr(f)),
               "mk_step_prepare")

    def launch(self):
        _check(lib.mk_step_launch(self.ctx), "mk_step_launch")

    def finish(self):
        out_t = np.zeros(self._nrows, np.int32)
        out_c = np.zeros(self._nseq, np.int32)
        _check(lib.mk_step_finish(self.ctx, _np_ptr(out_t), _np_ptr(out_c)), "mk_step_finish")
        return out_t[: int(out_c.sum())], out_c

    def last_drafts(self, n_seq: int):
        """MTP drafts of the last completed step: [n_seq][n_draft]."""
        d = np.zeros((n_seq, max(1, self.layout.n_draft)), np.int32)
        _check(lib.mk_last_drafts(self.ctx, _np_ptr(d)), "mk_last_drafts")
        return d

    def commit(self, seq_ids, n_keep):
        s = np.ascontiguousarray(seq_ids, np.int32)
        k = np.ascontiguousarray(n_keep, np.int32)
        _check(lib.mk_commit(self.ctx, len(s), _np_ptr(s), _np_ptr(k)), "mk_commit")

    def debug_outputs(self, logits=None, hidden=None):
        _check(lib.mk_debug_outputs(self.ctx, None if logits is None else logits.data_ptr(),
                                    None if hidden is None else hidden.data_ptr()), "mk_debug_outputs")

    def timeline(self, stamps=None):
        """Enable (int64 CUDA tensor of >= 5*n_layers+4 entries) or disable the phase timeline."""
        _check(lib.mk_debug_timeline(self.ctx, None if stamps is None else stamps.data_ptr()), "mk_debug_timeline")

    def skip_arrival(self, block: int, barrier: int, timeout_ns: int = 0):
        _check(lib.mk_debug_skip_arrival(self.ctx, block, barrier, timeout_ns), "mk_debug_skip_arrival")

    def scratch(self, rows: int):
        """Host copies of the last layer's scratch activations of the last step."""
        ys, os_ = i32(), i32()
        _check(lib.mk_debug_scratch(self.ctx, 0, None, None, None, None, ctypes.byref(ys), ctypes.byref(os_)),
               "mk_debug_scratch")
        m = self.model
        x = np.zeros((rows, m["hidden"]), np.float32)
        y = np.zeros((rows, ys.value), np.float32)
        o = np.zeros((rows, os_.value), np.float32)
        h = np.zeros((rows, m["ffn"]), np.float32)
        _check(lib.mk_debug_scratch(self.ctx, rows, _np_ptr(x), _np_ptr(y), _np_ptr(o), _np_ptr(h), None, None),
               "mk_debug_scratch")
        return dict(x=x.astype(np.float64), y=y.astype(np.float64), o=o.astype(np.float64),
                    h=h.astype(np.float64))

    def io_bytes(self):
        h, d = u64(), u64()
        _check(lib.mk_step_io_bytes(self.ctx, ctypes.byref(h), ctypes.byref(d)), "mk_step_io_bytes")
        return int(h.value), int(d.value)

    def last_launch_ms(self) -> float:
        return float(lib.mk_last_launch_ms(self.ctx))

    def grid_blocks(self) -> int:
        return int(lib.mk_grid_blocks(self.ctx))

    def close(self):
        if getattr(self, "ctx", None):
            lib.mk_free(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def q8_encode(x):
    """Test hook: the device q8 KV codec on a CUDA fp32 tensor of n x 32
    values (blocks of 32). Returns (codes int8 [n, 32], scales binary16 bits
    as int16 [n]) as CUDA tensors."""
    import torch
    x = x.contiguous().view(-1, 32)
    n = x.shape[0]
    q = torch.empty((n, 32), dtype=torch.int8, device=x.device)
    d = torch.empty((n,), dtype=torch.int16, device=x.device)
    stream = torch.cuda.current_stream(x.device).cuda_stream
    _check(lib.mk_debug_q8_encode(x.data_ptr(), n, q.data_ptr(), d.data_ptr(), stream), "mk_debug_q8_encode")
    return q, d


def attn_plan(q_rows_max: int, dh: int, q8: int):
    """Host-only test hook: the attention plan of a step (see mk_debug_attn_plan).
    Returns (status, dict)."""
    import numpy as np
    out = np.zeros(12, np.int32)
    rc = lib.mk_debug_attn_plan(q_rows_max, dh, q8, out.ctypes.data_as(vp))
    keys = ["nq", "jw", "wpg", "ng", "spg", "nslots", "xoff", "xslab", "phase_bytes", "slot_bytes",
            "ring_bytes", "page_list_bytes"]
    return rc, dict(zip(keys, (int(v) for v in out)))
