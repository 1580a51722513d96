"""Host logic of bench.py: rank aggregation (world size 2 over gloo), byte accounting."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    el, units = bench.combine_ranks(1.0 + rank, 100.0 * (rank + 1))
    out[rank] = (el, units)
    bench.barrier()
    dist.destroy_process_group()


def test_combine_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    # every rank sees the slowest rank's time and the tokens of all ranks
    assert out[0] == out[1] == (2.0, 300.0)


def test_combine_ranks_single_process():
    assert bench.combine_ranks(0.5, 64.0) == (0.5, 64.0)


def test_stage_bytes_by_hand():
    ids = np.array([[0, 1], [1, 2], [0, 1]])
    ad = np.array([0, -1, 0])
    st = bench.workload_stats(ids, ad, E=4)
    assert st == dict(T=3, k=2, S=6, E_touched=3, P=2, T_L=2, S_L=4)
    H, I, r, E = 8, 16, 4, 4
    b = bench.stage_bytes(st, H, I, E, r)
    # three experts' W1 (2I x H bf16), gathered rows in, fp32 rows out
    assert b["gate_up_gemm"] == 3 * 2 * I * H * 2 + 6 * H * 2 + 6 * 2 * I * 4
    # two (expert, adapter) pairs' A1 (r x H), two tokens' x rows, four slots' z
    assert b["gate_up_shrink"] == 2 * r * H * 2 + 2 * H * 2 + 4 * r * 4


def test_arguments():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "1"])


def test_host_info_fields():
    info = bench.host_info()
    assert isinstance(info["cpu_model"], str) and info["cpu_model"]
    assert set(info["blas"]) == {"library", "threads"}


def test_reference_arm_line(capsys):
    """The reference arm (the oracle on the host cores) prints one JSON line with the
    contract's keys; the tiny workload keeps it to a second."""
    import json
    assert bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "3",
                       "--warmup", "3"]) in (0, None)
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "impl", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 3 and d["value"] > 0
    assert d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["cpu_model"] and "threads" in cb["blas"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_launch_accounting_matches_the_plan():
    """gpu_launches counts kernels per layer call from the library's own plan (host only):
    with the expand fused into the grouped GEMMs, route (folded into the one-CTA align up
    to 64 tokens), align (one CTA; three kernels from 2048 slots), gather, two shrinks,
    two grouped GEMMs and the combine."""
    from types import SimpleNamespace
    import expert_adapter_gemms_gb300 as m
    from workloads import workload_by_name

    def count(name):
        c = workload_by_name(name)
        return bench.launches_per_layer(m, SimpleNamespace(**c))

    assert count("gptoss20b_decode") == 7
    assert count("gptoss20b_prefill") == 10
