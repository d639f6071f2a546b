"""The N>1 host path of bench.py on a real two-rank gloo group (CPU only):
distinct per-rank problems, max-over-ranks timing and the whole-job aggregate."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:  # the spawned ranks import this module afresh
    sys.path.insert(0, ROOT)


def free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from online_softmax_04_gb300 import workloads as wl

        w = wl.WORKLOADS[wl.HEADLINE]
        wr = bench.rank_workload(w, rank)
        ms = bench.max_over_ranks(10.0 * (rank + 1), dist, "cpu")
        value = bench.whole_job_tflops(world, bench.workload_flops(w), 7, ms)
        out[rank] = (wr.seed, ms, value)
    finally:
        dist.destroy_process_group()


def test_two_rank_gloo_aggregation():
    world = 2
    port = free_port()
    with mp.Manager() as m:
        out = m.dict()
        ctx = mp.get_context("spawn")
        procs = [ctx.Process(target=worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        res = dict(out)
    (s0, ms0, v0), (s1, ms1, v1) = res[0], res[1]
    assert s0 != s1                       # independent problems per rank
    assert ms0 == ms1 == 20.0             # both see the slowest rank
    import bench
    from online_softmax_04_gb300 import workloads as wl

    f = bench.workload_flops(wl.WORKLOADS[wl.HEADLINE])
    assert v0 == v1 == pytest.approx(2 * f * 7 / 0.020 / 1e12)


def test_single_process_helpers():
    import bench
    from online_softmax_04_gb300 import workloads as wl

    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    w = wl.WORKLOADS["B4-H16-N4096-d128-causal"]
    assert bench.workload_flops(w) == 4 * 4 * 16 * 4096 ** 2 * 128 / 2
    assert bench.rank_workload(w, 0).seed == w.seed


def test_step_stats():
    import bench

    assert bench.step_stats([]) is None
    assert bench.step_stats([3.0, 1.0, 2.0]) == {"min": 1.0, "median": 2.0, "max": 3.0, "n": 3}
    assert bench.step_stats([4.0, 1.0, 2.0, 3.0])["median"] == 2.5


def test_source_hash_ignores_comments():
    import bench

    code = 'int a = 1;\nconst char* s = "// kept /* kept */";\nchar q = \'"\';\n'
    with_comments = 'int a = 1; // one\n/* block\n comment */const char* s = "// kept /* kept */";\nchar q = \'"\'; // q\n'
    strip = bench.strip_c_comments
    assert strip(code) == code
    assert strip(with_comments).split() == strip(code).split()
    assert strip("int x; /* unterminated") == "int x;  "


def test_source_hash_ignores_comment_lines(tmp_path, monkeypatch):
    """Adding whole comment lines (and the blank lines they leave) keeps the hash; a code
    change does not."""
    import bench

    src = tmp_path / "online_softmax_04_gb300" / "csrc"
    src.mkdir(parents=True)
    f = src / "k.cuh"
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    f.write_text("int a = 1;\nint b = 2;\n")
    h0 = bench.kernel_source_hash("k")  # a kernel with no source list: every file counts
    f.write_text("// header\n//   more\nint a = 1;  // one\n\n// note\nint b = 2;\n")
    assert bench.kernel_source_hash("k") == h0
    f.write_text("int a = 1;\nint b = 3;\n")
    assert bench.kernel_source_hash("k") != h0


def test_forward_source_hash_covers_the_forward_files_only(tmp_path, monkeypatch):
    """The forward's traffic records lapse with a change to the files its kernels compile
    from, not with a change to the backward or row-softmax kernels."""
    import bench

    src = tmp_path / "online_softmax_04_gb300" / "csrc"
    src.mkdir(parents=True)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    for name in ("fa_fwd.cu", "fa_fwd_kernel.cuh", "fa_fwd_two_kernel.cuh", "sm103_ptx.cuh", "fa_bwd_kernel.cuh",
                 "softmax_rows.cuh"):
        (src / name).write_text(f"int {name.split('.')[0]} = 0;\n")
    h0 = bench.kernel_source_hash()
    (src / "fa_bwd_kernel.cuh").write_text("int changed = 1;\n")
    (src / "softmax_rows.cuh").write_text("int changed = 2;\n")
    assert bench.kernel_source_hash() == h0
    s0 = bench.kernel_source_hash("softmax_rows_smem")
    (src / "fa_fwd_two_kernel.cuh").write_text("int changed = 3;\n")
    assert bench.kernel_source_hash() != h0
    assert bench.kernel_source_hash("softmax_rows_smem") == s0
