"""The benchmark's byte accounting (the roofline's numerator), host only:
the 27B-shaped step streams 14.41 GB of Q4 weights, the cached K/V and the
recurrent state; an MTP head adds its weights, the draft lm_head rows and its
KV layer once per draft pass."""
import importlib.util
import os

from gen import configs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def test_weight_bytes_of_the_27b_step():
    b = _bench()
    ab = b.algorithmic_bytes(configs.QWEN27, 0, [(4096, 1)])
    assert abs(ab["weights"] / 1e9 - 14.41) < 0.01  # 25.62 G weights at 0.5625 B each, + one embedding row
    per_tok = 16 * 4 * 256 * 2 * 2  # 16 attention layers x 4 kv heads x dh x (K, V) x fp16
    assert ab["kv"] == (4096 + 1) * per_tok
    assert ab["total"] == ab["weights"] + ab["kv"] + ab["state"]


def test_mtp_passes_add_their_bytes():
    b = _bench()
    m = dict(configs.QWEN27, has_mtp=1, draft_vocab=32768)
    H, F = m["hidden"], m["ffn"]
    d = configs.model_dims(m)
    head = (H * 2 * H + (2 * d["fa_q"] + 2 * d["fa_kv"]) * H + H * d["fa_q"] + 3 * F * H) * 0.5625
    lm_rows = 32768 * H * 0.5625
    base = b.algorithmic_bytes(configs.QWEN27, 0, [(4096, 5)])
    for n_draft in (1, 4):
        ab = b.algorithmic_bytes(m, 0, [(4096, 5)], n_draft)
        extra_w = ab["weights"] - base["weights"]
        assert abs(extra_w - n_draft * (head + lm_rows + 5 * H * 0.5625)) < 1.0
        assert ab["kv"] - base["kv"] == n_draft * (4096 + 5) * 4 * 256 * 2 * 2
    # four passes: 1.33 GB, about 9 % of the step
    assert abs((ab["total"] - base["total"]) / 1e9 - 1.37) < 0.05


class _FakeWl:
    def __init__(self, seqs, vocab=100):
        import numpy as np
        self.seqs = seqs
        self.model = {"vocab": vocab}
        self.first_tokens = np.arange(7, 7 + len(seqs), dtype=np.int32)


def test_drafter_follows_trajectory_with_seeded_mismatch():
    """Each sequence's drafts copy its greedy trajectory up to the seeded
    mismatch position m, then differ: a greedy verifier accepts exactly m;
    advancing by the emitted count moves along the trajectory. Over many
    steps m is uniform over 0..T-1."""
    import numpy as np
    b = _bench()
    seqs = [(50, 3), (80, 3), (10, 3), (23, 3)]
    wl = _FakeWl(seqs)
    traj = [[(13 * s + 5 * j) % 100 for j in range(400)] for s in range(4)]
    d = b.Drafter(wl, traj, 2)
    seen = np.zeros(3, int)
    for step in range(60):
        tok, pos, sid = d.rows()
        at = 0
        out_t, out_c = [], []
        for s, (cached, T) in enumerate(seqs):
            rows = tok[at:at + T]
            assert list(sid[at:at + T]) == [s] * T
            assert list(pos[at:at + T]) == list(range(cached + d.off[s], cached + d.off[s] + T))
            assert rows[0] == d.last[s]
            o = d.off[s]
            a = 0  # greedy acceptance against the trajectory
            while a + 1 < T and rows[a + 1] == traj[s][o + a]:
                a += 1
            seen[a] += 1
            out_t += [int(x) for x in rows[1:a + 1]] + [traj[s][o + a]]
            out_c.append(a + 1)
            at += T
        before = list(d.off)
        d.advance(np.array(out_t), np.array(out_c))
        assert [d.off[s] - before[s] for s in range(4)] == out_c
    assert seen.min() > 0.2 * seen.sum() / 3  # every accept length occurs


def test_both_arms_share_the_config():
    b = _bench()
    a = b.workload_config("qwen27-4x3-23k-q8")
    assert a == b.workload_config("qwen27-4x3-23k-q8")
    assert a["rows_per_step"] == 12 and a["sequences"] == 4 and a["kv"] == "q8"
