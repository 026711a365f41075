"""The multi-rank path of bench.py on CPU: two gloo ranks, as torchrun starts
them (RANK / WORLD_SIZE / LOCAL_RANK / MASTER_* in the environment).

The layer shards over tokens, so the ranks are independent replicas: no
collective touches the data path. What the ranks share is host logic -- the
slowest replica's time is the job's time (a MAX all-reduce), the whole-job
throughput counts every replica's tokens, only rank 0 reports -- and the
inputs: the same parameters on every rank, their own tokens."""
import json
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402
from mixture_experts_layer_schedule_gb300 import inputs  # noqa: E402

WORLD = 2
SHAPE = inputs.LayerShape("mr", 64, 256, 512, 8, 2, zipf_s=1.2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out_dir):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(WORLD), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    ws_, r, local = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=ws_)
    cpu = torch.device("cpu")
    elapsed = 100.0 + 25.0 * rank  # rank 1 is the slow replica
    slowest = bench.max_over_ranks(elapsed, ws_, cpu)
    value = bench.replica_throughput(SHAPE.N, 10, ws_, slowest)
    inp = inputs.make_inputs(SHAPE, seed=rank, device="cpu", weight_seed=0)
    # every rank's parameters, and rank 0's view of the other rank's tokens
    w = torch.stack([inp["wg"].float().sum(), inp["wd"].float().sum(), inp["w_router"].float().sum()])
    ws_all = [torch.zeros_like(w) for _ in range(ws_)]
    dist.all_gather(ws_all, w)
    x_all = [torch.zeros(1) for _ in range(ws_)]
    dist.all_gather(x_all, inp["x"].float().sum().reshape(1))
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"ws": ws_, "local": local, "slowest": slowest, "value": value,
                   "same_params": all(torch.equal(ws_all[0], t) for t in ws_all),
                   "distinct_tokens": float(x_all[0]) != float(x_all[1])}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_replicas(tmp_path):
    mp.start_processes(_rank_main, args=(_free_port(), str(tmp_path)), nprocs=WORLD,
                       start_method="spawn", join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(WORLD)]
    for r, d in enumerate(res):
        assert d["ws"] == WORLD and d["local"] == r
        assert d["slowest"] == 125.0  # the MAX over ranks, on every rank
        assert d["value"] == pytest.approx(SHAPE.N * 10 * WORLD / 0.125)
        assert d["same_params"] and d["distinct_tokens"]


def test_single_rank_defaults(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.max_over_ranks(42.0, 1, None) == 42.0
    assert bench.replica_throughput(16384, 40, 1, 500.0) == pytest.approx(16384 * 40 / 0.5)
