"""The algorithmic work `bench.py` divides by (bytes and FLOPs per step),
checked against a brute-force enumeration of the keys every query token
sees on small seeded workloads (no GPU). The roofline fractions the bench
reports are only as right as these counts."""
import bench
from paged_latent_attention_cache_gb300 import workloads as W


def _brute(w):
    cs = w.cumseq.tolist()
    H, hs, vhs, bs, win = w.num_heads, w.head_size, w.v_head_size, w.block_size, w.local_window_size
    rows = flops = q_rows = bt = 0
    for b in range(w.num_seqs):
        seen = set()
        for t in range(cs[b], cs[b + 1]):
            pos = w.past_lens[b] + t - cs[b]
            keys = [j for j in range(pos + 1) if win < 0 or pos - j <= win]
            flops += len(keys) * H * (2 * hs + 2 * vhs)
            seen.update(keys)
            q_rows += 1
        rows += len(seen)
        bt += len({j // bs for j in seen})
    return rows, flops, q_rows, bt


def _check(w):
    got = bench.algorithmic_work(w, include_write=False)
    rows, flops, q_rows, bt = _brute(w)
    assert got["cache_rows"] == rows
    assert got["flops"] == flops
    assert got["tokens"] == q_rows
    el = 2
    el_c = 1 if w.cache_dtype == "e4m3" else 2   # an E4M3 cache row is hs bytes
    want = (rows * w.head_size * el_c + q_rows * w.num_heads * (w.head_size + w.v_head_size) * el +
            q_rows * w.rotary_dim * el + bt * 4)
    assert got["read_bytes"] == want


def test_accounting_causal():
    _check(W.make_workload("acc", q_lens=[1, 5, 0, 17], past_lens=[40, 0, 3, 9], num_heads=4,
                           **W.GLM, block_size=16, seed=3))


def test_accounting_window():
    _check(W.make_workload("accw", q_lens=[1, 30, 2], past_lens=[100, 50, 7], num_heads=2,
                           **W.GLM, block_size=16, seed=4, local_window_size=11))


def test_accounting_fp8_cache():
    _check(W.make_workload("acc8", q_lens=[1, 5, 0, 17], past_lens=[40, 0, 3, 9], num_heads=4,
                           **W.GLM, block_size=16, seed=6, cache_dtype="e4m3"))


def test_accounting_write_bytes():
    w = W.make_workload("accwr", q_lens=[3, 4], past_lens=[5, 0], num_heads=2, **W.GLM,
                        block_size=16, seed=5, drop_slots=2)
    a = bench.algorithmic_work(w)
    r = bench.algorithmic_work(w, include_write=False)
    written = int((w.slot_mapping >= 0).sum())
    assert written == w.num_tokens - 2
    el = 2
    assert a["bytes"] - r["bytes"] == (w.num_tokens * w.head_size * el +
                                       written * w.head_size * el +
                                       w.num_tokens * (w.rotary_dim * el + 4))


def test_accounting_separate_layout():
    """SEPARATE layout: a visible position is kv_num_heads key rows and
    kv_num_heads value rows."""
    w = W.make_separate_workload("accs", q_lens=[1, 5, 0, 17], past_lens=[40, 0, 3, 9],
                                 num_heads=8, kv_num_heads=2, head_size=64, block_size=16,
                                 seed=7)
    got = bench.algorithmic_work(w, include_write=False)
    rows, flops, q_rows, bt = _brute(w)
    assert got["cache_rows"] == rows and got["flops"] == flops
    want = (rows * 2 * (64 + 64) * 2 + q_rows * 8 * (64 + 64) * 2 + q_rows * w.rotary_dim * 2 +
            bt * 4)
    assert got["read_bytes"] == want
