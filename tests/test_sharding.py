"""The multi-rank path on CPU (gloo, world size 2): each rank generates and
verifies its own shard of a global batch with no data-path collective; the
shards together equal the whole batch, and the step time is the max over
ranks.  The GPU library is not involved (the oracle stands in for the
per-rank work, so the host-side sharding logic is what is tested)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, B, outdir):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import oracle
    import synth
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = synth.WORKLOADS["b8_k4_v32000_bf16"].with_(V=3000)
    inp = synth.generate(w, b0=rank * B, nb=B)
    res = oracle.load().verify(inp.logits, inp.q, inp.tokens, inp.u, inp.T)
    step_ms = torch.tensor([1.0 + rank])
    dist.all_reduce(step_ms, op=dist.ReduceOp.MAX)
    toks = torch.from_numpy(res.out_tokens.copy())
    gathered = [torch.empty_like(toks) for _ in range(world)]
    dist.all_gather(gathered, toks)  # test-side check only; not on the data path
    if rank == 0:
        np.save(os.path.join(outdir, "tokens.npy"), torch.cat(gathered).numpy())
        np.save(os.path.join(outdir, "step.npy"), step_ms.numpy())
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_shards_equal_whole_batch(tmp_path):
    import oracle
    import synth
    world, B = 2, 5
    mp.start_processes(_worker, args=(world, _free_port(), B, str(tmp_path)), nprocs=world,
                       start_method="spawn")
    w = synth.WORKLOADS["b8_k4_v32000_bf16"].with_(V=3000)
    whole = synth.generate(w, nb=world * B)
    ref = oracle.load().verify(whole.logits, whole.q, whole.tokens, whole.u, whole.T)
    got = np.load(tmp_path / "tokens.npy")
    assert np.array_equal(got, ref.out_tokens)
    assert float(np.load(tmp_path / "step.npy")[0]) == 2.0


def test_generator_shard_independence():
    import synth
    w = synth.WORKLOADS["b64_k5_v128256_bf16_topp"].with_(V=2000)
    whole = synth.generate(w, nb=6, nthreads=3)
    part = synth.generate(w, b0=2, nb=3, nthreads=1)
    assert np.array_equal(part.logits, whole.logits[2:5])
    assert np.array_equal(part.q, whole.q[2:5])
    assert np.array_equal(part.tokens, whole.tokens[2:5])
    assert np.array_equal(part.u, whole.u[2:5])
