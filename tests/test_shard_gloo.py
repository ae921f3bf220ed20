"""One scan split across ranks, host logic on CPU: gloo ranks run the partition and exchange of
selective_state_space_145_b300.shard with the fp64 oracle as every rank's compute, and the
gathered result must equal the oracle's unsharded scan of the whole problem.

The split by channel needs no exchange; the split by sequence segment exchanges each segment's
conv tail and its aggregate (sum of Delta, end state from zero) and composes them in order."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleBackend:
    """Every rank's compute through the fp64 oracle (CPU tensors in, float64 tensors out)."""

    def scan(self, x, delta, A, B, C, D, z, delta_bias, conv_w, conv_b, conv_init, h0):
        import oracle

        out, hl = oracle.selective_scan(x, delta, A, B, C, D, z, delta_bias, True, conv_w, conv_b, conv_init, h0)
        return torch.from_numpy(out), torch.from_numpy(hl)

    def aggregate(self, x, delta, A, B, delta_bias, conv_w, conv_b, conv_init):
        import oracle

        # S: the sum of Delta = softplus(delta + bias) over the segment; b: the end state from zero
        v = delta.double().numpy() + (0.0 if delta_bias is None else delta_bias.double().numpy()[None, :, None])
        S = oracle.softplus(v).sum(axis=2)
        _, hl = oracle.selective_scan(x, delta, A, B, B, None, None, delta_bias, True, conv_w, conv_b, conv_init,
                                      None)
        return torch.from_numpy(S), torch.from_numpy(hl)

    def compose(self, S, b, A, h0):
        import oracle

        A64 = A.double().numpy()
        h = np.zeros(b.shape[1:]) if h0 is None else h0.double().numpy()
        for j in range(S.shape[0]):
            a = np.exp(A64[None, :, :] * S[j].double().numpy()[:, :, None])
            _, h = oracle.compose(np.ones_like(a), h, a, b[j].double().numpy())
        return torch.from_numpy(h)


def _problem(seed):
    import sys

    sys.path.insert(0, ROOT)
    from selective_state_space_145_b300 import inputs

    return inputs.scan_inputs(2, 11, 53, 5, 4, "f32", seed=seed, with_h0=True, with_conv_init=True, random_A=True)


def _run(rank, world, port, q, mode, seg_lens):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from selective_state_space_145_b300 import shard

        p = _problem(seed=515)
        be = OracleBackend()
        if mode == "channels":
            out, hl = shard.scan_sharded_channels(p["x"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"],
                                                  p["delta_bias"], p["conv_w"], p["conv_b"], p["conv_init"], p["h0"],
                                                  backend=be)
        else:
            t0 = sum(seg_lens[:rank])
            t1 = t0 + seg_lens[rank]
            seg = lambda t: t[..., t0:t1].contiguous()
            out, hl = shard.scan_sharded_sequence(seg(p["x"]), seg(p["delta"]), p["A"], seg(p["B"]), seg(p["C"]),
                                                  p["D"], seg(p["z"]), p["delta_bias"], p["conv_w"], p["conv_b"],
                                                  p["conv_init"], p["h0"], backend=be)
        q.put((rank, out.numpy(), hl.numpy()))
    finally:
        dist.destroy_process_group()


def _spawn(world, mode, seg_lens=None):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_run, args=(r, world, port, q, mode, seg_lens)) for r in range(world)]
    for pr in procs:
        pr.start()
    res = dict((r, (o, h)) for r, o, h in (q.get(timeout=300) for _ in range(world)))
    for pr in procs:
        pr.join(timeout=120)
        assert pr.exitcode == 0
    return res


def _reference():
    import oracle

    p = _problem(seed=515)
    return oracle.selective_scan(p["x"], p["delta"], p["A"], p["B"], p["C"], p["D"], p["z"], p["delta_bias"], True,
                                 p["conv_w"], p["conv_b"], p["conv_init"], p["h0"])


def test_partition_tiles_the_range():
    from selective_state_space_145_b300.shard import partition

    for n in (0, 1, 5, 11, 1536):
        for world in (1, 2, 3, 8):
            parts = [partition(n, world, r) for r in range(world)]
            assert parts[0][0] == 0 and parts[-1][1] == n
            assert all(parts[r][1] == parts[r + 1][0] for r in range(world - 1))
            sizes = [b - a for a, b in parts]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        partition(4, 2, 2)


def test_channel_split_two_ranks_equals_the_whole_scan():
    ref, ref_h = _reference()
    res = _spawn(2, "channels")
    for r in range(2):  # every rank holds the gathered result
        out, hl = res[r]
        np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(hl, ref_h, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seg_lens", [[30, 23], [20, 2, 31]], ids=["two_ranks", "three_ranks_short_middle"])
def test_sequence_split_equals_the_whole_scan(seg_lens):
    """Segments in rank order, of unequal length; the middle one of the three-rank case is
    shorter than the conv window (d_conv - 1 = 3), so its window reaches into the segment before."""
    ref, ref_h = _reference()
    res = _spawn(len(seg_lens), "sequence", seg_lens)
    t0 = 0
    for r, n in enumerate(seg_lens):
        out, hl = res[r]
        np.testing.assert_allclose(out, ref[..., t0:t0 + n], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(hl, ref_h, rtol=1e-10, atol=1e-12)  # the final state, on every rank
        t0 += n
