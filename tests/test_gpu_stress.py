"""Repeated decode launches over long per-CTA block ranges (the TMA ring wraps
hundreds of times per CTA): no pipeline wait may give up (device status stays
0) and every launch must give bit-identical output."""
import pytest
import torch

from paged_kv_cache_252_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


@pytest.mark.parametrize("kv,D,Hq,n", [("fp16", 128, 32, 1), ("bf16", 128, 32, 1), ("e5m2", 128, 32, 1),
                                       ("fp16", 64, 32, 1), ("e5m2", 128, 64, 4), ("bf16", 128, 16, 2)])
def test_repeated_launches_are_clean_and_deterministic(dev, kv, D, Hq, n):
    import paged_kv_cache_252_gb300 as pkv
    w = wl.custom(num_seqs=4, num_q_heads=Hq, num_kv_heads=8, head_size=D, q_per_seq=n, kv_dtype=kv,
                  context_lens=[60000, 45000, 30001, 17], seed=99)
    vals = wl.token_values(w, device=dev)
    kc, vc = pkv.alloc_kv_cache(w.num_blocks, w.num_kv_heads, w.head_size, w.kv_dtype, dev)
    pkv.kv_cache_write(vals["k_all"], vals["v_all"], vals["slot_all"], kc, vc)
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    q = vals["q"]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ref = torch.empty_like(q)
    pkv.paged_attention_decode(ref, q, kc, vc, bt, cl, n, w.scale, device_status=status)
    out = torch.empty_like(q)
    for it in range(40):
        pkv.paged_attention_decode(out, q, kc, vc, bt, cl, n, w.scale, device_status=status)
        if it % 10 == 9:
            torch.cuda.synchronize()
            assert int(status.item()) == 0, f"device status {int(status.item()):#x} after {it + 1} launches"
            assert torch.equal(out, ref)
    assert torch.isfinite(ref).all()


def test_bounded_wait_gives_up_flags_and_leaves_the_context_usable(dev):
    """A wait on a barrier phase that nothing completes gives up after its limit and
    flags PKV_DEV_TIMEOUT; a second wait with the decode kernels' 2 s limit leaves on
    the CTA's abort flag; the next decode runs clean."""
    import paged_kv_cache_252_gb300 as pkv
    status, (t0, t1) = pkv.selftest_bounded_wait(2_000_000, dev)   # 2 ms
    assert status & 0x8
    assert 2_000_000 <= t0 < 200_000_000
    assert t1 < 200_000_000                                         # far below its own 2 s
    w = wl.custom(num_seqs=3, num_q_heads=8, num_kv_heads=2, head_size=128, q_per_seq=1, kv_dtype="fp16",
                  context_lens=[40, 300, 7], seed=3)
    import _gpu
    vals = wl.token_values(w)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    _gpu.cuda_path(w, vals, dev, status=st)
    assert int(st.item()) == 0
