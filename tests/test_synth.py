"""The seeded generators: deterministic, right shapes, right distributions."""
import numpy as np

import synth


def test_int4_problem_is_deterministic_and_shaped():
    a = synth.int4_problem(64, 256, seed=0)
    b = synth.int4_problem(64, 256, seed=0)
    c = synth.int4_problem(64, 256, seed=1)
    for key in ("qw", "s", "z", "x"):
        assert np.array_equal(a[key], b[key])
    assert not np.array_equal(a["qw"], c["qw"])
    assert a["qw"].shape == (64, 128) and a["qw"].dtype == np.uint8
    assert a["s"].shape == (64, 2) and a["z"].shape == (64, 2)
    assert a["x"].shape == (1, 256) and a["x"].dtype == np.uint16


def test_distributions():
    p = synth.int4_problem(512, 3840, seed=0)
    lo = p["qw"] & 15
    hi = p["qw"] >> 4
    for nib in (lo, hi):
        counts = np.bincount(nib.ravel(), minlength=16)
        assert counts.min() > 0.9 * nib.size / 16
    s = p["s"].view(np.float16).astype(np.float64)
    assert s.min() >= 0.002 - 1e-5 and s.max() <= 0.02 + 1e-5
    z = p["z"].view(np.float16).astype(np.float64)
    assert np.all(z == np.round(z)) and z.min() == 0 and z.max() == 15
    x = (p["x"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert abs(x.mean()) < 0.1 and abs(x.std() - 1.0) < 0.05


def test_expert_sampling_without_replacement():
    p = synth.fp4_moe_problem(64, 8, 64, topk=6, seed=0)
    ids = p["ids"]
    assert ids.dtype == np.int32 and len(set(ids.tolist())) == 6
    assert ids.min() >= 0 and ids.max() < 64
    seen = set()
    for seed in range(200):
        seen.update(synth.sample_experts(synth.Stream(seed), 64, 6).tolist())
    assert len(seen) == 64


def test_moe_batch_problem_routes_each_token_to_distinct_experts():
    p = synth.fp4_moe_batch_problem(E=16, N=8, K=64, M=5, topk=4, seed=3)
    q = synth.fp4_moe_batch_problem(E=16, N=8, K=64, M=5, topk=4, seed=3)
    assert p["ids"].shape == (5, 4) and p["x"].shape == (5, 64)
    assert all(len(set(row.tolist())) == 4 for row in p["ids"])
    assert p["ids"].min() >= 0 and p["ids"].max() < 16
    assert all(np.array_equal(p[k], q[k]) for k in ("qw", "s", "x", "ids"))
