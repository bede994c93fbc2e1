"""The q8 KV codec that the attention phase applies to the step's own K and V
rows (through the test hook mk_debug_q8_encode), against the oracle's codec,
which works in fp64, on identical fp32 inputs: every scale and every code
must be bit-exact.

The device computes the scale and the codes in single precision and corrects
them exactly (the neighbouring binary16 midpoints, the exact remainder), so
the cases that would expose a rounding slip are built in on purpose: max|x|
/ 127 exactly on a binary16 midpoint (a tie, to even) and one float step to
either side; codes exactly on half-integer ties (to even) and one float step
to either side; the clamp at +-127; zero blocks and blocks whose scale is a
binary16 subnormal; and random blocks of several magnitudes."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

from oracle import oracle as orc  # noqa: E402


def _h2f(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float32)


def _blocks():
    rng = np.random.default_rng(21)
    out = []
    # random blocks over many magnitudes
    for s in (1e-6, 1e-3, 0.02, 1.0, 37.0, 1e3):
        out.append((rng.standard_normal((64, 32)) * s).astype(np.float32))
    # amax / 127 on a binary16 midpoint (exact in fp32: 127 x a 12-bit value),
    # and one float step either side; even and odd lower neighbours
    for lo_bits in (0x2A00, 0x2A01, 0x3C00, 0x3C01, 0x0200, 0x0201, 0x5BFF):
        lo, hi = _h2f([lo_bits, lo_bits + 1])
        mid = np.float32(0.5) * (lo + hi)
        amax = np.float32(127) * mid
        for a in (amax, np.nextafter(amax, np.float32(np.inf)), np.nextafter(amax, np.float32(0))):
            b = np.clip(rng.standard_normal(32) * a / 4, -0.99 * a, 0.99 * a).astype(np.float32)
            b[3] = -a
            out.append(b[None])
    # codes on exact half-integer ties of the scale and one float step either side
    for d_bits in (0x2E66, 0x3800, 0x1A3F):
        d = _h2f([d_bits])[0]
        b = np.zeros((3, 32), np.float32)
        k = np.arange(-15, 16, dtype=np.float32)  # 31 ties k + 1/2 and the block max
        ties = (k + np.float32(0.5)) * d
        for r, f in enumerate((lambda v: v, lambda v: np.nextafter(v, np.float32(np.inf)),
                               lambda v: np.nextafter(v, np.float32(-np.inf)))):
            b[r, :31] = f(ties)
            b[r, 31] = np.float32(127) * d  # fixes the scale at d exactly
        out.append(b)
    # zero block, a block with one non-zero value, and values past the clamp
    z = np.zeros((1, 32), np.float32)
    one = np.zeros((1, 32), np.float32)
    one[0, 7] = np.float32(3.25)
    out += [z, one]
    return np.concatenate(out, 0).astype(np.float32)


def test_q8_codec_matches_oracle(cuda_ok):
    import torch
    from speculative_decode_persistent_gb300 import mk
    x = _blocks()
    q_gpu, d_gpu = mk.q8_encode(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    q_gpu = q_gpu.cpu().numpy()
    d_gpu = d_gpu.cpu().numpy().view(np.uint16)
    q_orc, d_orc = orc.q8_encode(x.astype(np.float64))
    bad = np.nonzero(d_gpu != d_orc)[0]
    assert bad.size == 0, [(int(i), float(np.abs(x[i]).max()), hex(d_gpu[i]), hex(d_orc[i])) for i in bad[:5]]
    badq = np.argwhere(q_gpu != q_orc)
    assert badq.size == 0, [(int(i), int(j), float(x[i, j]), int(q_gpu[i, j]), int(q_orc[i, j])) for i, j in badq[:5]]
    # the tie blocks did exercise both directions of round-half-even
    assert np.any(np.abs(q_orc) % 2 == 0) and np.any(np.abs(q_orc) % 2 == 1)


def test_q8_codec_empty_and_invalid(cuda_ok):
    import torch
    from speculative_decode_persistent_gb300 import mk
    q, d = mk.q8_encode(torch.zeros((0, 32), dtype=torch.float32, device="cuda"))
    assert q.shape == (0, 32) and d.shape == (0,)
    assert mk.lib.mk_debug_q8_encode(None, 4, None, None, None) == -1  # MK_ERR_INVALID
