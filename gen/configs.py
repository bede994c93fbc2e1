"""Model shapes, workloads and seeds of the verify-step configurations.

Pure data: sizes, seeds and the tensor inventory (names, ids, shapes) of the
canonical weight file layout. No arithmetic of the method lives here; both the
CPU oracle and the CUDA path read these numbers.

Sources: the hybrid decoder is the one the "Fusing the whole
speculative-decoding cycle into one CUDA kernel" page describes (64 layers, 48
Gated DeltaNet + 16 gated full attention, section "What shipped"); the exact
widths, head counts, vocabulary, contexts and draft depths are the workload
definitions this build was given (a tiny 4-layer model and the
Qwen3.8-27B-shaped model).
"""
from __future__ import annotations

import copy

GDN, FA = 0, 1

TINY = dict(
    name="tiny-4L-h256",
    n_layers=4,
    kinds=[GDN, GDN, GDN, FA],
    hidden=256,
    ffn=768,
    vocab=2048,
    hq=4, hkv=1, dh=64, rope_base=1e7,
    hk=2, hv=4, dk=64, dv=64, conv_w=4,
    tied=1,
    has_mtp=0, draft_vocab=0,
    eps=1e-6,
    weight_sigma=0.02,
)

QWEN27 = dict(
    name="qwen3.8-27b-shaped",
    n_layers=64,
    kinds=[GDN, GDN, GDN, FA] * 16,
    hidden=5120,
    ffn=17408,
    vocab=248320,
    hq=24, hkv=4, dh=256, rope_base=1e7,
    hk=16, hv=48, dk=128, dv=128, conv_w=4,
    tied=0,
    has_mtp=0, draft_vocab=0,
    eps=1e-6,
    weight_sigma=0.02,
)

PAGE_TOKENS = 16

# Workloads. "seqs" lists (cached tokens, rows this step) per sequence.
WORKLOADS = {
    "tiny": dict(model=TINY, kv_q8=0, n_pages=64, seqs=[(64, 4)], weight_seed=0,
                 cache_seed=1, draft_seed=2),
    "qwen27-t1-4k-fp16": dict(model=QWEN27, kv_q8=0, n_pages=320, seqs=[(4096, 1)],
                              weight_seed=0, cache_seed=1, draft_seed=2),
    "qwen27-t5-4k-fp16": dict(model=QWEN27, kv_q8=0, n_pages=320, seqs=[(4096, 5)],
                              weight_seed=0, cache_seed=1, draft_seed=2),
    "qwen27-t5-4k-fp16-mtp": dict(model=dict(QWEN27, has_mtp=1, draft_vocab=32768),
                                  kv_q8=0, n_pages=320, seqs=[(4096, 5)], n_draft=4,
                                  weight_seed=0, cache_seed=1, draft_seed=2),
    "qwen27-4x3-23k-q8": dict(model=QWEN27, kv_q8=1, n_pages=8448,
                              seqs=[(23000, 3)] * 4, shuffle_seed=3,
                              weight_seed=0, cache_seed=1, draft_seed=2),
    "qwen27-mixed-3x3-10k-q8+chunk512": dict(model=QWEN27, kv_q8=1, n_pages=8448,
                                             seqs=[(10000, 3)] * 3, chunk=(0, 512, 20000),
                                             weight_seed=0, cache_seed=1, prompt_seed=4),
    "qwen27-t5-96k-q8": dict(model=QWEN27, kv_q8=1, n_pages=6100, seqs=[(96000, 5)],
                             weight_seed=0, cache_seed=1, draft_seed=2),
}


def model_dims(m: dict) -> dict:
    """Derived widths of one model."""
    conv_ch = 2 * m["hk"] * m["dk"] + m["hv"] * m["dv"]
    return dict(
        conv_ch=conv_ch,
        gdn_out=m["hv"] * m["dv"],
        fa_q=m["hq"] * m["dh"],
        fa_kv=m["hkv"] * m["dh"],
        n_fa=sum(1 for k in m["kinds"] if k == FA),
        n_gdn=sum(1 for k in m["kinds"] if k == GDN),
    )


def tensor_inventory(m: dict) -> list[tuple[str, int, str, tuple]]:
    """Canonical tensors as (name, id, kind, shape); kind is "q4" or "f32".

    Q4 shapes are (rows, k) in weights; f32 shapes are element shapes.
    Ids key the generator streams: 1..3 global, 100*(layer+1)+slot per layer,
    and 9000+slot for the multi-token-prediction block.
    """
    H, F, V = m["hidden"], m["ffn"], m["vocab"]
    d = model_dims(m)
    out = [("embed", 1, "q4", (V, H)), ("final_norm", 2, "f32", (H,))]
    if not m["tied"]:
        out.append(("lm_head", 3, "q4", (V, H)))

    def block(prefix, base, kind):
        t = [(f"{prefix}.attn_norm", base + 0, "f32", (H,))]
        if kind == GDN:
            t += [
                (f"{prefix}.w_qkv", base + 1, "q4", (d["conv_ch"], H)),
                (f"{prefix}.w_z", base + 2, "q4", (d["gdn_out"], H)),
                (f"{prefix}.w_a", base + 3, "q4", (m["hv"], H)),
                (f"{prefix}.w_b", base + 4, "q4", (m["hv"], H)),
                (f"{prefix}.conv_w", base + 5, "f32", (d["conv_ch"], m["conv_w"])),
                (f"{prefix}.o_norm", base + 6, "f32", (m["dv"],)),
                (f"{prefix}.w_o", base + 20, "q4", (H, d["gdn_out"])),
            ]
        else:
            t += [
                (f"{prefix}.w_q", base + 11, "q4", (d["fa_q"], H)),
                (f"{prefix}.w_g", base + 12, "q4", (d["fa_q"], H)),
                (f"{prefix}.w_k", base + 13, "q4", (d["fa_kv"], H)),
                (f"{prefix}.w_v", base + 14, "q4", (d["fa_kv"], H)),
                (f"{prefix}.w_o", base + 20, "q4", (H, d["fa_q"])),
            ]
        t += [
            (f"{prefix}.ffn_norm", base + 21, "f32", (H,)),
            (f"{prefix}.w_gate", base + 22, "q4", (F, H)),
            (f"{prefix}.w_up", base + 23, "q4", (F, H)),
            (f"{prefix}.w_down", base + 24, "q4", (H, F)),
        ]
        return t

    for li, kind in enumerate(m["kinds"]):
        out += block(f"layers.{li}", 100 * (li + 1), kind)
    if m.get("has_mtp"):
        out += [
            ("mtp.norm_h", 9001, "f32", (H,)),
            ("mtp.norm_e", 9002, "f32", (H,)),
            ("mtp.fc", 9003, "q4", (H, 2 * H)),
            ("mtp.final_norm", 9004, "f32", (H,)),
        ]
        out += block("mtp.block", 9100, FA)
    return out


def with_overrides(name: str, **kw) -> dict:
    w = copy.deepcopy(WORKLOADS[name])
    w.update(kw)
    return w
