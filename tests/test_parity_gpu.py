"""GPU parity: the CUDA path through the C ABI against the CPU oracle on
the same seeded inputs, element by element.

Workloads: the tiny prefill+decode batch, GLM-style decode (H=64, 192/128,
batch 32, contexts U[1024, 8192]), DeepSeek-V3-style decode (H=128, 576/512,
batch 64, context 4096), DeepSeek-V3-style chunked prefill (4 x 4096 new
tokens over pasts {0,0,2048,2048}; outputs checked on a sample of tokens,
cache rows in full) and the mixed fp16 serving batch (window 4096,
softcap 50, 5% slots -1). Each runs on the default kernels (tensor-core where
specialised) and on the portable kernels.
"""
import numpy as np
import pytest
import torch

from tests import harness as Hn

pytestmark = pytest.mark.gpu

FULL = ["tiny", "glm_decode", "dsv3_decode", "mixed_serving"]


@pytest.fixture(scope="module")
def oracle_results():
    return {}


def _oracle(cache, name, tokens=None):
    key = (name, None if tokens is None else tuple(tokens))
    if key not in cache:
        cache[key] = Hn.run_oracle(Hn.workload(name), tokens)
    return cache[key]


@pytest.mark.parametrize("portable", [False, True], ids=["default", "portable"])
@pytest.mark.parametrize("name", FULL)
def test_workload_parity(name, portable, oracle_results):
    w = Hn.workload(name)
    got = Hn.run_gpu(w, portable=portable)
    ref = _oracle(oracle_results, name)
    assert got["flags"] == 0
    # the default path of every named workload is the tensor-core kernel
    expect = 0 if portable else 1
    assert got["op"].kernel_family(0) == expect and got["op"].kernel_family(1) == expect
    Hn.check_cache(w, got["cache"], ref["cache"])
    err, ratio = Hn.check_out(w, got["out"], ref["out"], scales=ref["scales"])
    print(f"RATIO {name} {'portable' if portable else 'default'}: max abs err {err:.3e}, "
          f"{ratio:.3f} of the scale-aware bound")


@pytest.mark.parametrize("portable", [False, True], ids=["default", "portable"])
def test_dsv3_prefill_parity_sampled(portable, oracle_results):
    w = Hn.workload("dsv3_prefill")
    tokens = Hn.sample_tokens(w, per_seq=16)
    got = Hn.run_gpu(w, portable=portable)
    ref = _oracle(oracle_results, "dsv3_prefill", tokens)
    assert got["flags"] == 0
    Hn.check_cache(w, got["cache"], ref["cache"])
    err, ratio = Hn.check_out(w, got["out"], ref["out"], tokens, ref["scales"])
    print(f"RATIO dsv3_prefill {'portable' if portable else 'default'}: max abs err {err:.3e}, "
          f"{ratio:.3f} of the scale-aware bound")


@pytest.mark.parametrize("gain", [8, 32])
@pytest.mark.parametrize("name", ["glm_decode", "dsv3_decode"])
def test_peaked_decode_parity(name, gain):
    """The full-size decode batches with the query scaled by 8 and 32: the
    logits spread over tens of units and the softmax is peaked, so errors in
    the scores (scale, rotation, the CTA pair's partial-score exchange) show
    in the outputs instead of averaging out over thousands of keys."""
    from paged_latent_attention_cache_gb300 import workloads as W
    w = W.peaked(Hn.workload(name), gain)
    got = Hn.run_gpu(w)
    ref = Hn.run_oracle(w)
    assert got["flags"] == 0
    assert got["op"].kernel_family(0) == 1
    err, ratio = Hn.check_out(w, got["out"], ref["out"], scales=ref["scales"])
    print(f"RATIO {w.name}: max abs err {err:.3e}, {ratio:.3f} of the scale-aware bound")


@pytest.mark.parametrize("name", ["glm_decode_fp8", "dsv3_decode_fp8"])
def test_fp8_cache_decode_parity(name, oracle_results):
    """GLM-style decode (H=64, 192/128, 32 sequences, contexts U[1024, 8192])
    and DeepSeek-style decode (H=128, 576/512, 64 x 4096) over an FP8 (E4M3)
    latent cache with k_scale = 1/64: the written codes are bit-exact outside
    the rotary channels and within one code inside; the outputs meet the
    bounds against the oracle of the FP8 operator."""
    w = Hn.workload(name)
    got = Hn.run_gpu(w)
    ref = _oracle(oracle_results, name)
    assert got["flags"] == 0
    assert got["op"].kernel_family(0) == 1
    Hn.check_cache(w, got["cache"], ref["cache"])
    err, ratio = Hn.check_out(w, got["out"], ref["out"], scales=ref["scales"])
    print(f"RATIO {name}: max abs err {err:.3e}, {ratio:.3f} of the scale-aware bound")


def test_single_key_rows_are_exact():
    """A token at position 0 sees only its own row: its output equals the
    written cache row's value channels exactly (the pages' "first token
    error exactly 0")."""
    from paged_latent_attention_cache_gb300 import workloads as W
    w = W.make_workload("first", q_lens=[3, 1], past_lens=[0, 0], num_heads=8, **W.GLM,
                        block_size=16, seed=11)
    got = Hn.run_gpu(w)
    vhs, hs = w.v_head_size, w.head_size
    cache = got["cache"].reshape(-1, hs)
    for t in (0, 3):
        row = cache[int(w.slot_mapping[t])]
        for h in range(w.num_heads):
            assert np.array_equal(got["out"][t, h * vhs:(h + 1) * vhs], row[:vhs])
