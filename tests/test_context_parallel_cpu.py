"""Key-sharded (context parallel) attention on the host: two gloo ranks each
attend to their own shard of the keys (the fp64 oracle stands in for the
per-shard kernel on CPU), exchange (o, lse) through the product's
``gather_partials``, and merge with the two-block rule (the oracle's
``softmax_merge``, CS149 Lecture 9 notes, concept 9).  The merged result must
equal attention over all keys.  The CUDA merge kernel itself is checked on
the GPU in test_merge_gpu.py."""
import os
import socket

import numpy as np
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        return so.getsockname()[1]


SPLIT = (37, 60)  # uneven shards of 97 keys


def _inputs():
    rng = np.random.default_rng(91)
    q = rng.standard_normal((1, 2, 5, 8))
    k = rng.standard_normal((1, 2, sum(SPLIT), 8))
    v = rng.standard_normal((1, 2, sum(SPLIT), 8))
    return q, k, v


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch
    import torch.distributed as dist

    import oracle
    from attention_flashattention_fwd_gb300.context_parallel import gather_partials
    dist.init_process_group("gloo", rank=rank, world_size=world)
    q, k, v = _inputs()
    k0 = sum(SPLIT[:rank])
    ks, vs = k[:, :, k0:k0 + SPLIT[rank]], v[:, :, k0:k0 + SPLIT[rank]]
    o, lse = oracle.attention(q, ks, vs, scale=0.5)
    o_parts, lse_parts = gather_partials(torch.tensor(o), torch.tensor(lse))
    out.put((rank, o_parts.numpy(), lse_parts.numpy()))
    dist.destroy_process_group()


def test_kv_sharded_attention_over_two_gloo_ranks():
    import oracle
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = {r: (o, l) for r, o, l in (out.get(timeout=120) for _ in procs)}
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    q, k, v = _inputs()
    ref_o, ref_lse = oracle.attention(q, k, v, scale=0.5)
    for rank in (0, 1):
        o_parts, lse_parts = res[rank]
        assert o_parts.shape == (2,) + ref_o.shape and lse_parts.shape == (2,) + ref_lse.shape
        # part s is rank s's shard, on every rank
        for s in (0, 1):
            k0 = sum(SPLIT[:s])
            o_s, l_s = oracle.attention(q, k[:, :, k0:k0 + SPLIT[s]], v[:, :, k0:k0 + SPLIT[s]],
                                        scale=0.5)
            assert np.array_equal(o_parts[s], o_s) and np.array_equal(lse_parts[s], l_s)
        # the merge of the gathered parts is attention over all keys
        for h in range(2):
            for i in range(5):
                m, l, o = oracle.softmax_merge(lse_parts[0, 0, h, i], 1.0, o_parts[0, 0, h, i],
                                               lse_parts[1, 0, h, i], 1.0, o_parts[1, 0, h, i])
                assert abs(m + np.log(l) - ref_lse[0, h, i]) <= 1e-12
                assert np.max(np.abs(o - ref_o[0, h, i])) <= 1e-13
