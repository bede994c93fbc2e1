"""ctypes front end of the fp64 CPU oracle (oracle/oracle.cpp).

TEST INFRASTRUCTURE ONLY: used by tests/, the smoke check and the CPU-baseline
leg of the benchmark. Shares no code with the CUDA library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_SO = os.path.join(_HERE, "liboracle.so")
_FLAGS = ["-O2", "-fPIC", "-shared", "-std=c++17", "-ffp-contract=off", "-pthread"]

i32, i64, dbl, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p


def build(force: bool = False) -> str:
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", *_FLAGS, "-o", tmp, _SRC])
        os.replace(tmp, _SO)
    return _SO


class OrcLayout(ctypes.Structure):
    _fields_ = [
        ("n_layers", i32), ("hidden", i32), ("ffn", i32), ("vocab", i32),
        ("kind", i32 * 64),
        ("hq", i32), ("hkv", i32), ("dh", i32), ("rope_base", dbl),
        ("hk", i32), ("hv", i32), ("dk", i32), ("dv", i32), ("conv_w", i32),
        ("tied", i32), ("has_mtp", i32), ("draft_vocab", i32), ("n_draft", i32),
        ("kv_q8", i32), ("page_tokens", i32), ("n_pages", i32), ("max_seqs", i32),
        ("max_pages_per_seq", i32),
        ("eps", dbl),
    ]


_LW = ["attn_norm", "w_qkv", "w_z", "w_a", "w_b", "conv_w", "o_norm", "w_q", "w_g", "w_k", "w_v",
       "w_o", "ffn_norm", "w_gate", "w_up", "w_down"]


class OrcLayerW(ctypes.Structure):
    _fields_ = [(n, vp) for n in _LW]


class OrcWeights(ctypes.Structure):
    _fields_ = [("embed", vp), ("final_norm", vp), ("lm_head", vp), ("layer", OrcLayerW * 64),
                ("mtp", OrcLayerW), ("mtp_fc", vp), ("mtp_norm_h", vp), ("mtp_norm_e", vp),
                ("mtp_final_norm", vp)]


class OrcPool(ctypes.Structure):
    _fields_ = [("k", vp), ("v", vp), ("kq", vp), ("vq", vp), ("ks", vp), ("vs", vp)]


_lib = None


def _bind(L):
    L.orc_create.restype = vp
    L.orc_create.argtypes = [ctypes.POINTER(OrcLayout), ctypes.POINTER(OrcWeights),
                             ctypes.POINTER(OrcPool), i32]
    L.orc_free.argtypes = [vp]
    L.orc_seq_set.argtypes = [vp, i32, i32, vp, i32, vp, vp]
    L.orc_seq_get.argtypes = [vp, i32, vp, vp, vp, vp, vp]
    L.orc_commit.argtypes = [vp, i32, vp, vp]
    L.orc_step.argtypes = [vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.orc_drafts.argtypes = [vp, i32, vp, vp, vp, vp, vp]
    L.orc_q4_decode.argtypes = [vp, i64, vp]
    L.orc_q4_encode.argtypes = [vp, i64, vp]
    L.orc_q4_matvec.argtypes = [vp, i32, i32, vp, vp, i32]
    L.orc_q8_encode.argtypes = [vp, i64, vp, vp]
    L.orc_sample_verify.argtypes = [vp, i32, i32, vp, dbl, i32, vp, vp]
    L.orc_sample_verify.restype = i32
    L.orc_half_round.argtypes = [dbl]
    L.orc_half_round.restype = ctypes.c_uint16
    L.orc_half_value.argtypes = [ctypes.c_uint16]
    L.orc_half_value.restype = dbl
    L.orc_rmsnorm.argtypes = [vp, vp, i32, dbl, vp]
    L.orc_l2norm.argtypes = [vp, i32, dbl]
    L.orc_rope.argtypes = [vp, i32, i32, dbl]
    L.orc_attend.argtypes = [vp, vp, vp, i32, i32, vp]
    L.orc_gdn_update.argtypes = [vp, i32, i32, vp, vp, vp, dbl, dbl, vp]
    L.orc_sigmoid.argtypes = [dbl]
    L.orc_sigmoid.restype = dbl
    L.orc_silu.argtypes = [dbl]
    L.orc_silu.restype = dbl
    L.orc_n_free_pages.argtypes = [vp]
    for f in ("orc_seq_set", "orc_seq_get", "orc_commit", "orc_step", "orc_n_free_pages", "orc_drafts"):
        getattr(L, f).restype = ctypes.c_int
    return L


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(_SO))
    return _lib


def build_variant(substitutions: list[tuple[str, str]], out_dir: str):
    """A copy of the oracle with each (old, new) source substitution applied
    (each `old` must occur exactly once), compiled into out_dir and loaded.
    Tests use it to plant a known mistake and check that a pin catches it."""
    with open(_SRC) as f:
        src = f.read()
    for old, new in substitutions:
        n = src.count(old)
        if n != 1:
            raise ValueError(f"substitution target occurs {n} times: {old!r}")
        src = src.replace(old, new)
    os.makedirs(out_dir, exist_ok=True)
    cpp = os.path.join(out_dir, "oracle_variant.cpp")
    so = os.path.join(out_dir, "liboracle_variant.so")
    with open(cpp, "w") as f:
        f.write(src)
    subprocess.check_call(["g++", *_FLAGS, "-o", so, cpp])
    return _bind(ctypes.CDLL(so))


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "contiguous numpy array expected"
    return a.ctypes.data_as(vp)


def make_layout(model: dict, kv_q8: int, n_pages: int, max_seqs: int, page_tokens: int = 16,
                max_pages_per_seq: int | None = None, n_draft: int = 0) -> OrcLayout:
    L = OrcLayout()
    L.n_layers, L.hidden, L.ffn, L.vocab = model["n_layers"], model["hidden"], model["ffn"], model["vocab"]
    for i, k in enumerate(model["kinds"]):
        L.kind[i] = k
    L.hq, L.hkv, L.dh, L.rope_base = model["hq"], model["hkv"], model["dh"], model["rope_base"]
    L.hk, L.hv, L.dk, L.dv, L.conv_w = model["hk"], model["hv"], model["dk"], model["dv"], model["conv_w"]
    L.tied, L.has_mtp, L.draft_vocab, L.n_draft = model["tied"], model.get("has_mtp", 0), model.get("draft_vocab", 0), n_draft
    L.kv_q8, L.page_tokens, L.n_pages, L.max_seqs = kv_q8, page_tokens, n_pages, max_seqs
    L.max_pages_per_seq = max_pages_per_seq or n_pages
    L.eps = model["eps"]
    return L


class Oracle:
    """fp64 CPU model step over numpy-held weights and a numpy-held KV pool."""

    def __init__(self, model: dict, weights: dict, pool: dict, kv_q8: int, n_pages: int,
                 max_seqs: int, nthreads: int | None = None, n_draft: int = 0, library=None):
        self._lib = library if library is not None else lib()
        self.model = model
        self._keep = [weights, pool]
        self.L = make_layout(model, kv_q8, n_pages, max_seqs, n_draft=n_draft)
        W = OrcWeights()
        W.embed = _p(weights["embed"])
        W.final_norm = _p(weights["final_norm"])
        W.lm_head = _p(weights["lm_head"]) if "lm_head" in weights else None
        for li in range(model["n_layers"]):
            for n in _LW:
                key = f"layers.{li}.{n}"
                if key in weights:
                    setattr(W.layer[li], n, _p(weights[key]))
        if model.get("has_mtp"):
            for n in _LW:
                key = f"mtp.block.{n}"
                if key in weights:
                    setattr(W.mtp, n, _p(weights[key]))
            W.mtp_fc = _p(weights["mtp.fc"])
            W.mtp_norm_h = _p(weights["mtp.norm_h"])
            W.mtp_norm_e = _p(weights["mtp.norm_e"])
            W.mtp_final_norm = _p(weights["mtp.final_norm"])
        P = OrcPool()
        for n in ("k", "v", "kq", "vq", "ks", "vs"):
            if n in pool:
                setattr(P, n, _p(pool[n]))
        self.W, self.P = W, P
        self.nthreads = int(nthreads or os.cpu_count() or 1)
        self.h = self._lib.orc_create(ctypes.byref(self.L), ctypes.byref(W), ctypes.byref(P), self.nthreads)
        if not self.h:
            raise ValueError("orc_create rejected the layout")

    def __del__(self):
        if getattr(self, "h", None):
            self._lib.orc_free(self.h)
            self.h = None

    # dims
    @property
    def n_gdn(self):
        return sum(1 for k in self.model["kinds"] if k == 0)

    @property
    def conv_ch(self):
        m = self.model
        return 2 * m["hk"] * m["dk"] + m["hv"] * m["dv"]

    def seq_set(self, seq: int, length: int, pages, S=None, conv=None):
        pages = np.ascontiguousarray(pages, dtype=np.int32)
        S = None if S is None else np.ascontiguousarray(S, dtype=np.float32)
        conv = None if conv is None else np.ascontiguousarray(conv, dtype=np.float32)
        rc = self._lib.orc_seq_set(self.h, seq, length, _p(pages), len(pages), _p(S), _p(conv))
        if rc:
            raise ValueError(f"orc_seq_set failed ({rc})")

    def seq_get(self, seq: int):
        m = self.model
        length, npg = ctypes.c_int(0), ctypes.c_int(0)
        pages = np.zeros(self.L.n_pages, np.int32)
        S = np.zeros((self.n_gdn, m["hv"], m["dv"], m["dk"]), np.float64)
        conv = np.zeros((self.n_gdn, m["conv_w"] - 1, self.conv_ch), np.float64)
        rc = self._lib.orc_seq_get(self.h, seq, ctypes.byref(length), _p(pages), ctypes.byref(npg), _p(S), _p(conv))
        if rc:
            raise ValueError("orc_seq_get failed")
        return dict(length=length.value, pages=pages[: npg.value].copy(), S=S, conv=conv)

    def commit(self, seq_ids, n_keep):
        s = np.ascontiguousarray(seq_ids, np.int32)
        k = np.ascontiguousarray(n_keep, np.int32)
        rc = self._lib.orc_commit(self.h, len(s), _p(s), _p(k))
        if rc:
            raise ValueError(f"orc_commit failed ({rc})")

    def step(self, tokens, positions, seq_ids, flags=None, want_logits=True, want_hidden=False):
        tokens = np.ascontiguousarray(tokens, np.int32)
        positions = np.ascontiguousarray(positions, np.int32)
        seq_ids = np.ascontiguousarray(seq_ids, np.int32)
        R = len(tokens)
        fl = None if flags is None else np.ascontiguousarray(flags, np.uint8)
        nseq = len({int(s) for s in seq_ids})
        out_tokens = np.zeros(R, np.int32)
        out_counts = np.zeros(nseq, np.int32)
        logits = np.zeros((R, self.model["vocab"]), np.float64) if want_logits else None
        hidden = np.zeros((R, self.model["hidden"]), np.float64) if want_hidden else None
        argmax = np.zeros(R, np.int32)
        gap = np.zeros(R, np.float64)
        rms = np.zeros(R, np.float64)
        rc = self._lib.orc_step(self.h, R, _p(tokens), _p(positions), _p(seq_ids), _p(fl),
                            _p(out_tokens), _p(out_counts), _p(logits), _p(hidden), _p(argmax),
                            _p(gap), _p(rms))
        if rc:
            raise ValueError(f"orc_step failed ({rc})")
        n_out = int(out_counts.sum())
        return dict(tokens=out_tokens[:n_out], counts=out_counts, logits=logits, hidden=hidden,
                    argmax=argmax, gap=gap, rms=rms)

    def drafts(self, seq: int):
        """Drafts of the sequence's last verify step (model with a
        multi-token-prediction block and n_draft > 0)."""
        m, n = self.model, self.L.n_draft
        d = np.zeros(n, np.int32)
        gap = np.zeros(n, np.float64)
        rms = np.zeros(n, np.float64)
        logits = np.zeros((n, m["draft_vocab"]), np.float64)
        hidden = np.zeros((n, m["hidden"]), np.float64)
        rc = self._lib.orc_drafts(self.h, seq, _p(d), _p(gap), _p(rms), _p(logits), _p(hidden))
        if rc:
            raise ValueError(f"orc_drafts failed ({rc})")
        return dict(tokens=d, gap=gap, rms=rms, logits=logits, hidden=hidden)

    def n_free_pages(self):
        return self._lib.orc_n_free_pages(self.h)


# ------------------------------------------------------------------ blocks

def q4_decode(blocks: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(blocks, np.uint8).reshape(-1, 144)
    out = np.zeros(b.shape[0] * 256, np.float64)
    lib().orc_q4_decode(_p(b), b.shape[0], _p(out))
    return out


def q4_encode(w: np.ndarray) -> np.ndarray:
    w = np.ascontiguousarray(w, np.float64).reshape(-1, 256)
    out = np.zeros((w.shape[0], 144), np.uint8)
    lib().orc_q4_encode(_p(w), w.shape[0], _p(out))
    return out


def q4_matvec(W: np.ndarray, K: int, u: np.ndarray, nthreads: int = 1) -> np.ndarray:
    W = np.ascontiguousarray(W, np.uint8)
    rows = W.shape[0]
    u = np.ascontiguousarray(u, np.float64)
    y = np.zeros(rows, np.float64)
    lib().orc_q4_matvec(_p(W), rows, K, _p(u), _p(y), nthreads)
    return y


def q8_encode(x: np.ndarray):
    x = np.ascontiguousarray(x, np.float64).reshape(-1, 32)
    q = np.zeros(x.shape, np.int8)
    d = np.zeros(x.shape[0], np.uint16)
    lib().orc_q8_encode(_p(x), x.shape[0], _p(q), _p(d))
    return q, d


def sample_verify(logits: np.ndarray, drafts, temperature: float, top_k: int, u: np.ndarray, library=None):
    """Speculative sampling verification of one sequence's rows (see
    orc_sample_verify): logits [T][V], drafts [T-1], u [T][2] uniforms in
    [0, 1). Returns the emitted tokens (accepted drafts, then the last one).
    library: a variant built by build_variant (tests), else the oracle."""
    logits = np.ascontiguousarray(logits, np.float64)
    T, V = logits.shape
    d = np.ascontiguousarray(np.asarray(drafts, np.int32).reshape(-1))
    u = np.ascontiguousarray(u, np.float64).reshape(T, 2)
    out = np.zeros(T, np.int32)
    L = library if library is not None else lib()
    n = L.orc_sample_verify(_p(logits), T, V, _p(d) if T > 1 else None, float(temperature), int(top_k),
                            _p(u), _p(out))
    if n < 0:
        raise ValueError("orc_sample_verify: bad argument")
    return [int(x) for x in out[:n]]


def half_round(x: float) -> int:
    return int(lib().orc_half_round(float(x)))


def half_value(h: int) -> float:
    return float(lib().orc_half_value(int(h)))


def rmsnorm(x, g, eps):
    x = np.ascontiguousarray(x, np.float64)
    g = None if g is None else np.ascontiguousarray(g, np.float32)
    y = np.zeros_like(x)
    lib().orc_rmsnorm(_p(x), _p(g), len(x), eps, _p(y))
    return y


def l2norm(x, eps):
    x = np.array(x, np.float64)
    lib().orc_l2norm(_p(x), len(x), eps)
    return x


def rope(x, pos, base):
    x = np.array(x, np.float64)
    lib().orc_rope(_p(x), len(x), pos, base)
    return x


def attend(q, K, V):
    q = np.ascontiguousarray(q, np.float64)
    K = np.ascontiguousarray(K, np.float64)
    V = np.ascontiguousarray(V, np.float64)
    out = np.zeros(K.shape[1], np.float64)
    lib().orc_attend(_p(q), _p(K), _p(V), K.shape[0], K.shape[1], _p(out))
    return out


def gdn_update(S, q, k, v, alpha, beta):
    """Returns (new S, o). S is dv x dk."""
    S = np.array(S, np.float64)
    dv, dk = S.shape
    o = np.zeros(dv, np.float64)
    lib().orc_gdn_update(_p(S), dk, dv, _p(np.ascontiguousarray(q, np.float64)),
                         _p(np.ascontiguousarray(k, np.float64)), _p(np.ascontiguousarray(v, np.float64)),
                         alpha, beta, _p(o))
    return S, o


def sigmoid(v):
    return lib().orc_sigmoid(float(v))


def silu(v):
    return lib().orc_silu(float(v))
