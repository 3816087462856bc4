"""Host-side logic of bench.py on CPU: the multi-rank timing reduction over
gloo (world size 2), the reference arm's JSON line, and the workload recipes."""

import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from exact_io_aware_107_b300 import workloads as W  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    try:
        _rank_body(rank, world, port, q)
    except BaseException as e:  # report instead of leaving the peer waiting
        q.put((rank, "error", repr(e)))
        raise


def _rank_body(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, local = bench.dist_env()
    bench.barrier(ws)
    m = bench.max_over_ranks(1.5 + rank, ws)     # rank 1 is the slow one
    # the reference arm runs on rank 0 only; rank 1 exits without output
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--workload", "f32_causal_b2_h4_n128_d64",
                         "--steps", "1", "--warmup", "3"])
    dist.destroy_process_group()
    q.put((rank, ws, r, local, m, rc, buf.getvalue()))


def test_two_rank_gloo_reduction_and_reference_arm():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted((q.get(timeout=240) for _ in procs), key=lambda t: t[0])
    assert all(t[1] != "error" for t in out), out
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, ws0, rr0, l0, m0, rc0, txt0), (r1, ws1, rr1, l1, m1, rc1, txt1) = out
    assert ws0 == ws1 == 2 and (rr0, rr1) == (0, 1) and (l0, l1) == (0, 1)
    assert m0 == m1 == 2.5                         # max over ranks
    assert rc0 == rc1 == 0
    line = json.loads(txt0.strip())
    assert txt1.strip() == ""
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1


def test_reference_arm_single_process():
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.main(["--impl", "reference", "--workload", "f32_causal_b2_h4_n128_d64",
                           "--steps", "2", "--warmup", "1"]) == 0
    line = json.loads(buf.getvalue().strip())
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["warmup"] == 3          # at least three warm-up steps are enforced
    assert line["config"]["workload"] == "f32_causal_b2_h4_n128_d64"
    assert line["unit"] == "TFLOP/s" and line["higher_is_better"] is True


def test_flop_counts():
    w = W.WORKLOADS["bf16_causal_b2_h32_n8192_d128"]
    assert w.flops() == 4 * 2 * 32 * 8192 ** 2 * 128 / 2
    v = W.WORKLOADS["bf16_varlen_causal_h32_d128"]
    assert v.flops() == sum(4 * 32 * L * L * 128 for L in v.varlen) / 2
    assert W.WORKLOADS["bf16_b4_h16_n2048_d64"].flops() == 4 * 4 * 16 * 2048 ** 2 * 64


def test_generators_are_seeded_and_rounded():
    w = W.custom("bf16", B=1, H=2, N=33, D=64, seed=5)
    a, b = W.generate(w), W.generate(w)
    for key in ("q", "k", "v"):
        assert a[key].dtype == b[key].dtype
        assert (a[key].float() == b[key].float()).all()
    # bf16 values widen to fp64 exactly: the low 16 bits of the fp32 pattern are zero
    bits = a["q"].float().numpy().view(np.uint32)
    assert (bits & 0xFFFF == 0).all()
    # the small fp32 case follows the legacy global-generator call sequence
    f = W.generate(W.WORKLOADS["f32_causal_b2_h4_n128_d64"])
    np.random.seed(0)
    np.testing.assert_array_equal(f["q"].numpy(),
                                  np.random.randn(2, 4, 128, 64).astype(np.float32))


def test_varlen_lengths_from_seed_7():
    v = W.WORKLOADS["bf16_varlen_causal_h32_d128"]
    assert len(v.varlen) == 16 and all(256 <= L <= 8192 for L in v.varlen)
    cu = W.cu_seqlens_of(v.varlen)
    assert cu[0] == 0 and cu[-1] == v.N and (np.diff(cu) > 0).all()


@pytest.mark.parametrize("name", sorted(W.WORKLOADS))
def test_workload_config_keys(name):
    cfg = bench.workload_config(W.WORKLOADS[name])
    assert cfg["workload"] == name and cfg["flops_per_step"] > 0


def test_cross_flop_counts_follow_the_pair_count():
    # 4*D flops per allowed (query, key) pair; the causal count drops the
    # diagonal's half pair per row, as the self-attention N^2/2 convention does
    for nq, nk, causal in ((2048, 8192, True), (8192, 1024, False), (300, 77, True),
                           (77, 300, True)):
        w = W.custom("bf16", B=2, H=3, N=nq, D=64, causal=causal, Nk=nk)
        i = np.arange(nq)
        exact = np.clip(i + 1 + nk - nq, 0, nk).sum() if causal else nq * nk
        assert abs(w.flops() - 4 * 64 * 6 * exact) <= 4 * 64 * 6 * (nq / 2 + 1e-9)
    w = W.CROSS_WORKLOADS["bf16_cross_causal_b2_h32_nq2048_nk8192_d128"]
    assert w.flops() == 4 * 128 * 64 * (2048 * 8192 - 2048 ** 2 / 2)


def test_cross_generator_shapes():
    w = W.custom("bf16", B=2, H=3, N=40, D=64, Nk=70, seed=1)
    x = W.generate(w)
    assert tuple(x["q"].shape) == (2, 3, 40, 64) and tuple(x["k"].shape) == (2, 3, 70, 64)
    assert tuple(x["v"].shape) == (2, 3, 70, 64)
    p = W.generate(W.custom("f32", H=2, D=16, varlen=[3, 0, 5], varlen_k=[4, 2, 0]))
    assert tuple(p["q"].shape) == (2, 8, 16) and tuple(p["k"].shape) == (2, 6, 16)
    assert list(p["cu_seqlens"]) == [0, 3, 3, 8] and list(p["cu_seqlens_k"]) == [0, 4, 6, 6]
    # with Nk == N the draw is the self-attention draw
    a = W.generate(W.custom("bf16", B=1, H=2, N=33, D=64, seed=5))
    b = W.generate(W.custom("bf16", B=1, H=2, N=33, D=64, seed=5, Nk=33))
    for key in ("q", "k", "v"):
        assert (a[key].float() == b[key].float()).all()


@pytest.mark.parametrize("name", sorted(W.CROSS_WORKLOADS))
def test_cross_workload_config_keys(name):
    cfg = bench.workload_config(W.CROSS_WORKLOADS[name])
    assert cfg["workload"] == name and cfg["Nk"] == W.CROSS_WORKLOADS[name].n_keys


def test_oracle_units_cover_every_plane_and_cap_long_ones():
    w = W.custom("bf16", B=2, H=3, N=40, D=64, seed=3)
    units = bench._oracle_units(w, W.generate(w))
    assert len(units) == 6 and all(u[0].shape == (40, 64) for u in units)
    v = W.custom("bf16", H=2, D=64, varlen=[5, 9000, 3], seed=4)
    units = bench._oracle_units(v, W.generate(v))
    # one unit per (sequence, head); the long sequence keeps its last rows, all keys
    assert [u[0].shape[0] for u in units] == [5, 5, bench.UNIT_ROWS, bench.UNIT_ROWS, 3, 3]
    assert units[2][1].shape[0] == 9000


def test_unit_flops_count_allowed_pairs():
    q, k = np.zeros((3, 8)), np.zeros((5, 8))
    # last 3 queries of a 5-key causal plane see 3, 4 and 5 keys
    assert bench._unit_flops(q, k, True, 8) == 4 * 8 * (3 + 4 + 5)
    assert bench._unit_flops(q, k, False, 8) == 4 * 8 * 15
    assert bench._unit_flops(k, k, True, 8) == 4 * 8 * 15


def test_host_cores_respects_the_affinity_mask():
    n = bench.host_cores()
    assert 1 <= n <= len(os.sched_getaffinity(0))
    q = bench.cgroup_cpu_limit()
    assert q is None or q >= 1


def test_cpu_baseline_on_a_small_workload():
    # the process pool (spawned workers) and the one-process figure
    w = W.WORKLOADS["f32_causal_b2_h4_n128_d64"]
    x = W.generate(w)
    r = bench.cpu_baseline(w, x, cpu_seconds=0.5)
    assert r["kind"] == "oracle" and r["value"] > 0 and r["value_1core"] > 0
    assert 1 <= r["cores"] <= bench.host_cores()
    assert "oracle.attention_plane" in r["sample"] and "whole planes" in r["sample"]
