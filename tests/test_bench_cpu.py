"""bench.py's algorithmic work accounting (CPU): flops and bytes of a layer-step follow
from the visible lengths the oracle defines."""
import numpy as np

import bench
import oracle.mla_ref as R
import synth


def test_work_matches_oracle_lengths():
    for name, lengths in [("tiny", None), ("cp2", None), ("spec", [100, 2345]),
                          ("long", [5000, 4097])]:
        w = synth.make_workload(name, lengths=lengths)
        wk = bench.work(w)
        G = w.G.numpy()
        flops = 0.0
        kv_rows = 0
        for r in range(w.cp):
            sl = R.ref_local_len(G, w.cp, r)
            kv_rows += int(sl.sum())
            for b in range(w.B):
                for i in range(w.q_len):
                    Gi = int(R.ref_row_global_prefix(G[b], w.q_len)[i])
                    Li = min(int(sl[b]), int(R.ref_local_len(Gi, w.cp, r)))
                    flops += w.H * 2 * (576 + 512) * Li
        assert kv_rows == int(G.sum())
        assert abs(wk["flops"] - flops) < 1e-6 * max(flops, 1)
        assert wk["kv_bytes"] == float(G.sum() * 1152)
        assert wk["q_bytes"] == float(w.cp * w.B * w.q_len * w.H * 1152)


def test_cpu_baseline_sample_is_bounded():
    r = bench.cpu_baseline_sample("tiny", budget_s=0.5)
    assert r["kind"] == "oracle" and r["value"] > 0 and r["cores"] >= 1
    assert "requests" in r["sample"]
