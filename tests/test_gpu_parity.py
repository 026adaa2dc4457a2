"""GPU path vs the fp64 oracle on the seeded workloads, through the C ABI.

Attention outputs must satisfy |gpu - oracle| <= 2e-3 + 1e-2 |oracle|
element by element; the cache state after the step's copies and writes must
be bit-identical to the oracle's for every block the step touches, and every
other byte of the pools must still be the poison pattern.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
import synth.device as SD
import synth.host as H
from gpu_helpers import assert_close, device_error, run_step, sample_pools, to_f64, oracle_outputs
from synth.device import to_storage

pytestmark = pytest.mark.gpu

THREADS = max(1, min(16, len(os.sched_getaffinity(0))))


def _bits(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint32) if a.dtype == np.float32 else a


def _check_pools(dw, hp, kc_ref, vc_ref, what):
    idx = torch.from_numpy(hp.ids).to(dw.k_cache.device)
    for dev_pool, ref in ((dw.k_cache, kc_ref), (dw.v_cache, vc_ref)):
        got = to_storage(dev_pool[idx])
        assert np.array_equal(_bits(got), _bits(ref)), f"{what}: cache bytes differ from the oracle"
        # every byte outside those blocks is still poison
        words = dev_pool.view(torch.int32)
        touched_live = int((_bits(ref).view(np.int32) != -1).sum())
        assert int((words != -1).sum().item()) == touched_live, f"{what}: bytes outside the step changed"


SMALL = [
    ("tiny", None, {}),
    ("llama7b", 8, {}),
    ("llama13b", 8, {}),
    ("cow", 12, {}),
    ("longctx_bs8", 2, {"num_heads": 4, "num_kv_heads": 4}),
    ("longctx_bs16", 2, {"num_heads": 4, "num_kv_heads": 4}),
    ("longctx_bs32", 2, {"num_heads": 4, "num_kv_heads": 4}),
]


@pytest.mark.parametrize("name,B,over", SMALL, ids=[s[0] for s in SMALL])
def test_small_workload(name, B, over):
    cfg = synth.get(name).replace(**over)
    hw = H.generate(cfg, num_seqs=B)
    hp = H.compact_pools(hw)
    dw = SD.from_host(hw)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_step(dw, dev_err=err)
    assert device_error(err) == 0
    ref, kc_ref, vc_ref = oracle.decode_step(hp, hw, threads=THREADS)
    assert_close(to_f64(out), ref, name)
    _check_pools(dw, hp, kc_ref, vc_ref, name)
    del dw
    torch.cuda.empty_cache()


FULL = ["llama7b", "llama13b", "cow", "longctx_bs8", "longctx_bs16", "longctx_bs32"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload(name):
    """The full workloads, in the launch configuration the benchmark times;
    every output element is checked against the oracle."""
    cfg = synth.get(name)
    dw = SD.generate(cfg)
    hp = sample_pools(dw, np.arange(dw.st.num_seqs))  # host copy before any kernel runs
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = run_step(dw, dev_err=err)
    assert device_error(err) == 0
    got = to_f64(out)
    assert np.isfinite(got).all()
    ref = oracle_outputs(dw, hp, threads=THREADS)
    stats = assert_close(got, ref, name)
    print(f"{name}: {stats}")
    _check_pools(dw, hp, hp.k_cache, hp.v_cache, name)  # decode_step updated hp's pools in place
    del dw
    torch.cuda.empty_cache()
