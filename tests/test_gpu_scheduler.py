"""The multi-agent host scheduler on the CUDA engine (tiny model): three
agents, two of them starting with a shared prefix that is processed once and
copied (KV pages and recurrent state, Engine.clone_sequence), with
prompt-lookup drafts and stacked, chunked rows; every conversation's greedy
text must equal the fp64 oracle running it alone, one token per step, and a
follow-up request continues in the same slot."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

from gen.workload import Workload  # noqa: E402
from oracle import oracle as orc  # noqa: E402
from test_scheduler import oracle_solo  # noqa: E402


def test_scheduler_on_the_engine(cuda_ok):
    from speculative_decode_persistent_gb300 import mk
    from speculative_decode_persistent_gb300.scheduler import AgentScheduler
    wl = Workload("tiny", nthreads=4)

    def make():
        return orc.Oracle(wl.model, wl.weights, {k: v.copy() for k, v in wl.pool.items()}, wl.kv_q8,
                          wl.n_pages, wl.max_seqs, nthreads=4)

    eng = mk.Engine(wl.model, wl.weights, wl.kv_q8, wl.n_pages, max_seqs=wl.max_seqs)
    eng.load_pool(wl.pool)
    rng = np.random.default_rng(19)
    V = wl.model["vocab"]
    system = [int(x) for x in rng.integers(0, V, 21)]
    users = [[int(x) for x in rng.integers(0, V, n)] for n in (3, 11)]
    other = [int(x) for x in rng.integers(0, V, 9)] * 2
    sch = AgentScheduler(eng, n_draft=2)
    sch.register_prefix(system)
    for i, u in enumerate(users):
        sch.submit(i, system + u, 8)
    sch.submit("other", other, 8)
    out = sch.run()
    for i, u in enumerate(users):
        assert out[i] == oracle_solo(make, system + u, 8), i
    assert out["other"] == oracle_solo(make, other, 8)
    slot = sch.convs[0].slot
    more = [int(x) for x in rng.integers(0, V, 4)]
    sch.submit(0, more, 6)
    out2 = sch.run()
    assert sch.convs[0].slot == slot
    assert out2[0] == oracle_solo(make, system + users[0] + out[0] + more, 6)
    eng.close()
