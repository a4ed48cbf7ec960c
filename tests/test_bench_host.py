"""Host-side logic of bench.py: the replicated (weak-scaling) aggregation across ranks,
run as two gloo processes on the CPU, and the clock-sample summary."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        el, units = bench.aggregate(1.0 + rank, 100.0 * (rank + 1), world)
        bench.barrier(world)
        q.put((rank, el, units))
    finally:
        torch.distributed.destroy_process_group()


def test_aggregate_takes_max_time_and_total_units_over_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, el, units in res:
        assert el == 2.0 and units == 300.0


def test_single_rank_aggregate_is_identity():
    assert bench.aggregate(0.5, 7.0, 1) == (0.5, 7.0)


def test_clock_summary():
    lines = ["0, 2070, 2070, 300.5, 0x0, Not Active, Not Active, Not Active, Not Active",
             "0, 1900, 2070, 900.0, 0x4, Not Active, Not Active, Not Active, Active",
             "0, 2070, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "garbage"]
    s = bench.summarize_clocks(lines)
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 950.0
    assert bench.summarize_clocks([]) is None


def test_warmup_floor():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_reference_arm_reports_the_same_config():
    """Both arms describe the workload with one function, so their `config`
    objects are identical for the same workload, L2 size and rank count."""
    from paged_kv_cache_252_gb300 import workloads as wl
    for key in ("8b", "70b_spec", "long"):
        w = wl.by_name(key)
        l2 = 126 << 20
        pools = bench.pool_count(w, l2)
        assert pools >= 2 and pools * w.kv_bytes_read() > 4 * l2
        a = bench.bench_config(w, pools, l2, 1)
        b = bench.bench_config(wl.by_name(key), bench.pool_count(wl.by_name(key), l2), l2, 1)
        assert a == b and a["workload"] == w.name and "l2_policy" in a


def test_product_source_drops_only_profiling_hooks():
    """The traffic digest covers the source the product library compiles: the
    PKV_TIMELINE branches and PKV_TL* hook lines go, their #else branches and all
    other preprocessor blocks stay."""
    text = ("a();\n"
            "#ifdef PKV_TIMELINE\n  t0 = clock64();\n  if (!got) {\n#else\n  if (x) {\n#endif\n"
            "  if (tid == 0) PKV_TL_STEP(3);\n"
            "#if defined(OTHER)\n  b();\n#else\n  c();\n#endif\n"
            "#ifdef PKV_TIMELINE\n  only_profiling();\n#endif\n"
            "d();\n")
    assert bench.product_source(text) == ("a();\n  if (x) {\n#if defined(OTHER)\n  b();\n#else\n  c();\n#endif\n"
                                          "d();\n")
    # a change outside the hooks changes the digest input
    assert bench.product_source(text.replace("d();", "e();")) != bench.product_source(text)
