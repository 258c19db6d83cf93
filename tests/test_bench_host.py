"""Host-side logic of bench.py: the multi-rank reduction on world_size-2 gloo ranks (the
data path has no collective; only the timing is reduced), the reference arm's JSON
line on the tiny workload, and the source digest that keys the ncu counters."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = bench.max_over_ranks(1.0 + rank, world, "cpu")
    v = bench.job_throughput(world, 10, 100.0, t)
    dist.destroy_process_group()
    out.put((rank, t, v))


def test_max_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.0, 2.0]          # slowest rank's time everywhere
    assert [r[2] for r in res] == [1000.0, 1000.0]    # 2 ranks x 10 steps x 100 units / 2 s


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(1, 4, 10.0, 2.0) == 20.0


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "cpu_baseline", "e2e", "config"):
        assert key in line, key
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"


def test_source_digest_ignores_comments_but_not_code():
    """The counters' source digest follows the compiled code: comment and layout edits keep
    it, any code edit (including inside a string literal) changes it."""
    import bench
    src = 'int a = 1; // note\n/* block\n comment */ const char *s = "x // y";\n'
    assert bench._code_only(src) == bench._code_only(src.replace("note", "other").replace("\n", "\n\n"))
    assert bench._code_only(src) != bench._code_only(src.replace("a = 1", "a = 2"))
    assert bench._code_only(src) != bench._code_only(src.replace("x // y", "x // z"))


def test_source_digest_covers_the_fused_kernels_translation_unit():
    """The digest lists exactly the files the fused kernel is compiled from."""
    import bench
    tu = bench.kernel_includes(os.path.join(ROOT, "stem_ssb_phase_gb300", "csrc", "ssb_fused.cu"))
    assert sorted(os.path.relpath(f, ROOT) for f in tu) == sorted(bench.KERNEL_SOURCES)


def test_redraw_and_upsample_byte_counts():
    """The algorithmic bytes the redraw and interpolation rooflines divide by."""
    import bench
    # G cache of the full workload: 8,937 planes of 257 x 512 complex64
    assert bench.redraw_algorithmic_bytes(8937, 512) == 9_407_729_664
    # interpolation at f = 4: float64 accumulator in, 2048^2 float32 phase + complex64 out
    assert bench.upsample_algorithmic_bytes(512, 4) == 512 * 512 * 16 + 2048 * 2048 * 12
    assert bench.upsample_algorithmic_bytes(512, 1, want_object=False) == 512 * 512 * 20
