"""Gated attention at the 27B-shaped head geometry (24 q heads, 4 kv heads,
head dim 256) against the fp64 oracle: one attention layer over long cached
contexts in fp16 and q8 pools, for one sequence at T = 1 and T = 5 and for
four sequences at T = 3 on a shuffled page pool. A small vocabulary and FFN
keep the oracle fast; the attention work is full size.

Every test drives the CUDA path through the C ABI (libmk.so via ctypes)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

from helpers import Pair  # noqa: E402
from gen import configs  # noqa: E402


def _model():
    return dict(configs.QWEN27, n_layers=1, kinds=[configs.FA], vocab=4096, ffn=512)


CASES = {
    # name: (seqs, shuffled pages)
    "t1-3000": ([(3000, 1)], False),
    "t5-2500": ([(2500, 5)], False),
    "4x3-ragged": ([(1500, 3), (777, 3), (2049, 3), (16, 3)], True),
    "t8-short": ([(40, 8)], False),
}


@pytest.mark.parametrize("kv_q8", [0, 1])
@pytest.mark.parametrize("case", list(CASES))
def test_attention_27b_heads(cuda_ok, kv_q8, case):
    seqs, shuffle = CASES[case]
    n_pages = sum((c + T + 15) // 16 for c, T in seqs) + 8
    ov = dict(model=_model(), kv_q8=kv_q8, n_pages=n_pages, seqs=seqs)
    if shuffle:
        ov["shuffle_seed"] = 3
    p = Pair("qwen27-t1-4k-fp16", overrides=ov, nthreads=8)
    wl = p.wl
    rng = np.random.default_rng(5)
    tok, pos, sid = wl.rows([list(rng.integers(0, wl.model["vocab"], T - 1)) for (_c, T) in seqs])
    ro, rg = p.step(tok, pos, sid)
    p.compare_step(ro, rg, sid)
    for s in range(len(seqs)):
        p.compare_kv(s, [int(x) for x, q in zip(pos, sid) if q == s])


@pytest.mark.parametrize("kv_q8", [0, 1])
def test_attention_27b_heads_prompt_rows(cuda_ok, kv_q8):
    """Eight prompt rows ending the prompt (flags 1 x 7, then 2) over a
    2,000-token cache: causal over the rows, no verification, one token."""
    seqs = [(2000, 8)]
    ov = dict(model=_model(), kv_q8=kv_q8, n_pages=(2000 + 8 + 15) // 16 + 8, seqs=seqs)
    p = Pair("qwen27-t1-4k-fp16", overrides=ov, nthreads=8)
    tok = np.array(np.random.default_rng(13).integers(0, p.wl.model["vocab"], 8), np.int32)
    pos = np.arange(2000, 2008, dtype=np.int32)
    sid = np.zeros(8, np.int32)
    flags = np.array([1] * 7 + [2], np.uint8)
    ro, rg = p.step(tok, pos, sid, flags)
    p.compare_step(ro, rg, sid, flags)
    assert list(rg["counts"]) == [1]
    p.compare_kv(0, pos.tolist())


def test_attention_27b_heads_96k_q8(cuda_ok):
    """The long-context workload's attention at full size: T = 5 rows over a
    96,000-token q8 cache (about 38 splits of 158 pages per kv head, merged by
    all of a head's split blocks), against the oracle."""
    seqs = [(96000, 5)]
    ov = dict(model=_model(), kv_q8=1, n_pages=(96000 + 5 + 15) // 16 + 8, seqs=seqs)
    p = Pair("qwen27-t1-4k-fp16", overrides=ov, nthreads=16)
    rng = np.random.default_rng(17)
    tok, pos, sid = p.wl.rows([list(rng.integers(0, p.wl.model["vocab"], 4))])
    ro, rg = p.step(tok, pos, sid)
    p.compare_step(ro, rg, sid)
    p.compare_kv(0, [int(x) for x in pos])
