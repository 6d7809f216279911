"""Host-side logic of bench.py and the workload generator (CPU only), including
the multi-rank timing reduction over a world-size-2 gloo process group."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workloads


def test_flop_convention():
    # forward 2 N^2 (d_qk + d_v), backward 2 N^2 (3 d_qk + 2 d_v); causal counts half the square
    assert workloads.attn_flops(8192, 8192, 128, 128, False, "fwd") == 2 * 8192 ** 2 * 256
    assert workloads.attn_flops(8192, 8192, 128, 128, True, "fwd") == 8192 ** 2 * 256
    assert workloads.attn_flops(100, 100, 192, 128, False, "bwd") == 2 * 100 ** 2 * (3 * 192 + 2 * 128)
    w = workloads.Workload("x", 4, 16, 8192, 8192, 128, 128, False)
    f = bench.step_flops(w)
    assert f[("fwd", True)] * 2 == f[("fwd", False)]
    assert f[("bwd", False)] == 2.5 * f[("fwd", False)]
    assert abs(sum(f.values()) - 4 * 16 * (2.2e12 / 64) * 0 - sum(f.values())) == 0


def test_varlen_flops_sum_over_sequences():
    w = workloads.varlen_32seq()
    assert sum(w.varlen_lengths) == 498963
    expect = 32 * sum(2 * n * n / 2 * 256 for n in w.varlen_lengths)
    assert abs(workloads.workload_flops(w, "fwd") - expect) < 1e-6 * expect


def test_generator_is_seeded_and_bf16():
    w = workloads.single_head_d64()
    a, b = workloads.make_dense(w), workloads.make_dense(w)
    for n in ("q", "k", "v", "do"):
        assert a[n].dtype == torch.bfloat16 and torch.equal(a[n], b[n])
    c = workloads.make_dense(w.with_(seed=1))
    assert not torch.equal(a["q"], c["q"])


def test_outlier_rows_are_scaled():
    w = workloads.dense_d128(1024, False, outlier=True).with_(batch=1, heads=2)
    base = workloads.make_dense(w.with_(outlier_frac=0.0), with_do=False)["k"].float()
    out = workloads.make_dense(w, with_do=False)["k"].float()
    changed = (base != out).any(dim=-1)  # [B, N, H]
    assert changed.sum(dim=1).tolist() == [[11, 11]]  # ceil(1% of 1024) rows per (batch, head)


def test_sample_pairs_deterministic_and_in_range():
    p = workloads.sample_pairs(4, 16, 5, seed=3)
    assert p == workloads.sample_pairs(4, 16, 5, seed=3)
    assert len(set(p)) == 5 and all(0 <= b < 4 and 0 <= h < 16 for b, h in p)


def test_reduce_max_without_process_group():
    assert bench.reduce_max(3.5) == 3.5


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, wsz, local = bench.dist_env()
    assert (r, wsz, local) == (rank, world, rank)
    bench.barrier()
    out[rank] = bench.reduce_max(10.0 + rank)
    dist.destroy_process_group()


def test_multi_rank_timing_reduction_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: 11.0, 1: 11.0}


def test_bench_rejects_short_warmup():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "1"])


def test_causal_pair_count_matches_brute_force():
    import workloads
    for nq, nk in [(2048, 8192), (8192, 2048), (5, 3), (3, 5), (1, 1000), (1000, 1), (513, 700)]:
        brute = sum(min(max(i + nk - nq + 1, 0), nk) for i in range(nq))
        assert workloads.causal_pairs(nq, nk) == brute
    assert workloads.causal_pairs(8192, 8192) == 8192 * 8192 / 2  # the half-square convention


def test_traffic_key_ignores_comments_only():
    """The roofline's traffic figures stay valid across documentation edits of the
    kernel sources, and go null on any code change."""
    import bench
    a = 'int x = 1; // one\n/* block\n comment */\nconst char* s = "a // b";\n\n  y = x;  \n'
    b = 'int x = 1;\nconst char* s = "a // b";\n  y = x;\n// trailing\n'
    c = 'int x = 2;\nconst char* s = "a // b";\n  y = x;\n'
    assert bench.code_only(a) == bench.code_only(b)
    assert bench.code_only(a) != bench.code_only(c)
    assert '"a // b"' in bench.code_only(a)
    for k in bench.KERNEL_SOURCES:
        assert len(bench.kernel_sources_sha(k)) == 16
