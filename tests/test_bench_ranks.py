"""The benchmark's multi-rank host logic on CPU with gloo, world size 2:
rendezvous, barrier, max-over-ranks timing, distinct per-rank workloads and the
whole-job value.  (Every box here has one GPU; the GPU ranks run the same code
over NCCL.)"""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    import gen

    w_, r_, l_ = bench.dist_setup()
    assert (w_, r_) == (world, rank)
    t = bench.max_over_ranks(1.0 + rank, world, torch.device("cpu"))
    bench.barrier(world)
    seed = bench.replica_seed("llama3_8b", rank)
    wl = gen.make("llama3_8b", B=4, lens=("uniform", 1, 64), max_len=64, seed=seed)
    with open(os.path.join(out_dir, "r%d.txt" % rank), "w") as f:
        f.write("%r %d %s\n" % (t, seed, ",".join(map(str, wl.lens_np.tolist()))))
    import torch.distributed as dist

    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    rows = [open(tmp_path / ("r%d.txt" % r)).read().split() for r in range(world)]
    assert all(float(r[0]) == 2.0 for r in rows)         # max over ranks
    assert rows[0][1] != rows[1][1]                       # distinct replica seeds
    assert rows[0][2] != rows[1][2]                       # hence distinct workloads


@pytest.mark.timeout(300)
def test_gpus_flag_starts_that_many_ranks():
    """`bench.py --gpus 2` outside a launcher starts two ranks under
    torch.distributed.run (gloo on CPU); the reference arm's rank 0 prints the
    one JSON line, with n_gpus 2, and the other rank exits without work."""
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    res = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2",
                          "--impl", "reference", "--config", "tiny", "--steps", "3",
                          "--warmup", "3", "--cpu-threads", "1"],
                         capture_output=True, text=True, cwd=root, env=env, timeout=280)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [json.loads(x) for x in res.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, res.stdout
    assert lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2


def test_gpus_flag_must_match_the_launcher():
    """Under a launcher that started one rank, `--gpus 2` is refused instead of
    printing a one-GPU line as if it were two."""
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    res = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2",
                          "--impl", "reference", "--config", "tiny", "--steps", "3",
                          "--warmup", "3"], capture_output=True, text=True, cwd=root, env=env,
                         timeout=120)
    assert res.returncode == 2 and "--gpus 2" in res.stderr
    assert not res.stdout.strip()


def test_relaunch_command():
    import bench

    cmd = bench.relaunch_cmd(["--gpus", "4", "--steps", "9"], 4, 29555)
    i = cmd.index("torch.distributed.run")
    assert cmd[i - 1] == "-m" and cmd[cmd.index("--nproc-per-node") + 1] == "4"
    assert cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"
    assert cmd[cmd.index("--master-port") + 1] == "29555"
    assert cmd[-4:] == ["--gpus", "4", "--steps", "9"] and cmd[-5].endswith("bench.py")


def test_whole_job_value():
    import bench

    assert bench.whole_job_gbs(nbytes=1e9, t_ms=2.0, world=4) == pytest.approx(2000.0)


def test_reference_arm_reports_its_core_count():
    """`--impl reference --cpu-threads 1` times the oracle on one host core and
    says so; without the flag it uses every core OpenMP offers."""
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--config",
           "tiny", "--steps", "3", "--warmup", "3"]
    one = json.loads(subprocess.run(cmd + ["--cpu-threads", "1"], capture_output=True, text=True,
                                    check=True, cwd=root).stdout.strip().splitlines()[-1])
    assert one["impl"] == "reference" and one["cpu_baseline"]["cores"] == 1
    assert "1 host core" in one["cpu_baseline"]["sample"] and one["value"] > 0


def test_kernel_hash_tracks_code_not_comments(tmp_path):
    """The committed DRAM-traffic counters are reported only while the decode
    kernel's code is the code they were taken on: an edit of comments or
    whitespace keeps bench.kernel_hash(), any code edit changes it."""
    import shutil

    import bench

    src = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                       "paged_gqa_decode_04_gb300", "csrc")
    work = tmp_path / "csrc"
    shutil.copytree(src, work)
    base = bench.kernel_hash(str(work))
    assert base == bench.kernel_hash(src)
    cuh = work / "decode_tma.cuh"
    text = cuh.read_text()
    cuh.write_text("// a new comment line\n" + text.replace("\n\n", "\n\n\n", 3))
    assert bench.kernel_hash(str(work)) == base
    cuh.write_text(text.replace("kMinTilesPerCta = 2;", "kMinTilesPerCta = 3;"))
    assert bench.kernel_hash(str(work)) != base
    cuh.write_text(text)
    (work / "partition.cuh").write_text((work / "partition.cuh").read_text() + "\nint x;\n")
    assert bench.kernel_hash(str(work)) != base
    # a string literal is code: a "//" inside one is not a comment
    (work / "partition.cuh").write_text((work / "partition.cuh").read_text().replace(
        "int x;", 'const char* s = "a // b";'))
    h1 = bench.kernel_hash(str(work))
    (work / "partition.cuh").write_text((work / "partition.cuh").read_text().replace(
        '"a // b"', '"a // c"'))
    assert bench.kernel_hash(str(work)) != h1
