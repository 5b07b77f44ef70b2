"""Expert-parallel split on CPU ranks (gloo, world size 2): the partition of the
experts, the decode schedule (one sum all-reduce of y) and the prefill schedule
(all-to-all dispatch of rows to their experts' owners, all-to-all combine of the
partial outputs).  The per-rank compute here is the CPU oracle restricted to a
rank's experts, so the host logic of routed_expert_decode_gb300.expert_parallel
is checked against the single-rank oracle layer: expert indices and offsets
exact, y within the layer's 1e-3 normwise tolerance."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))
for p in (ROOT, TESTS):
    if p not in sys.path:
        sys.path.insert(0, p)

import oracle  # noqa: E402
import synth  # noqa: E402
from routed_expert_decode_gb300.expert_parallel import (ExpertParallel, expert_ranges,  # noqa: E402
                                                        owner_of)

SPEC = synth.LayerSpec("ep_small", E=16, k=4, d=256, f=128, f_shared=128, fmt=0, s=2.5,
                       zipf_beta=0.4)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def oracle_partial(spec, experts, shared, bias):
    """The oracle layer restricted to routed experts [lo, hi) and, if
    with_shared, the shared expert: shared first, then the owned slots in slot
    order, fp64 sums of the oracle's expert rows, fp32 routing weights."""

    def partial(x, logits, lo, hi, with_shared):
        xn, ln = x.numpy(), logits.numpy()
        idx, w = oracle.route(ln, bias, spec.k, spec.s, score=spec.score)
        y = np.zeros((xn.shape[0], spec.d), np.float64)
        for t in range(xn.shape[0]):
            xq, xs = oracle.quantize(xn[t])
            if with_shared and spec.f_shared:
                y[t] += oracle.expert_row(oracle.FMT_Q8_0, spec.d, spec.f_shared, shared, xq, xs)[2]
            for j in range(spec.k):
                e = int(idx[t, j])
                if lo <= e < hi:
                    y[t] += float(w[t, j]) * oracle.expert_row(spec.fmt, spec.d, spec.f,
                                                               experts[e], xq, xs)[2]
        return torch.from_numpy(y.astype(np.float32))

    return partial


def oracle_route(spec, bias):
    def route(logits):
        idx, _ = oracle.route(logits.numpy(), bias, spec.k, spec.s, score=spec.score)
        return torch.from_numpy(idx.astype(np.int64))

    return route


def _layer_inputs(spec):
    experts = {e: synth.expert_host(spec, e) for e in range(spec.E)}
    shared = synth.expert_host(spec, spec.E) if spec.f_shared else None
    return experts, shared, synth.bias(spec)


def _reference(spec, experts, shared, bias, x, logits):
    return oracle.layer(spec.E, spec.k, spec.d, spec.f, spec.f_shared, spec.fmt, spec.s,
                        experts, shared, x, logits, bias)


def _normwise(a, b):
    return float((np.abs(a - b).max(axis=1) / np.abs(b).max(axis=1)).max())


def test_expert_ranges_partition():
    for E, world in ((16, 2), (256, 8), (192, 3), (7, 7), (10, 4)):
        r = expert_ranges(E, world)
        assert r[0][0] == 0 and r[-1][1] == E
        assert all(r[i][1] == r[i + 1][0] for i in range(world - 1))
        sizes = [hi - lo for lo, hi in r]
        assert max(sizes) - min(sizes) <= 1
        for e in range(E):
            lo, hi = r[owner_of(e, r)]
            assert lo <= e < hi
    with pytest.raises(ValueError):
        expert_ranges(3, 4)


def test_single_rank_schedules_equal_the_layer():
    """world = 1: decode and prefill reduce to the whole layer (the prefill
    exchanges become copies)."""
    experts, shared, bias = _layer_inputs(SPEC)
    logits, x = synth.token_inputs(SPEC, 3, 6)
    ep = ExpertParallel(SPEC.E, 0, 1, oracle_partial(SPEC, experts, shared, bias),
                        oracle_route(SPEC, bias))
    ref = _reference(SPEC, experts, shared, bias, x, logits)
    for y in (ep.decode(torch.from_numpy(x), torch.from_numpy(logits)),
              ep.prefill(torch.from_numpy(x), torch.from_numpy(logits))):
        assert _normwise(y.numpy(), ref.y) <= 1e-3


def _worker(rank, world, port, mode, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        experts, shared, bias = _layer_inputs(SPEC)
        ep = ExpertParallel(SPEC.E, rank, world, oracle_partial(SPEC, experts, shared, bias),
                            oracle_route(SPEC, bias))
        # decode: every rank the same tokens; prefill: each rank its own
        T = 5 if mode == "decode" else 7 + 2 * rank
        seed = 40 if mode == "decode" else 50 + rank
        logits, x = synth.token_inputs(SPEC, seed, T)
        if mode == "decode":
            y = ep.decode(torch.from_numpy(x), torch.from_numpy(logits))
        else:
            y = ep.prefill(torch.from_numpy(x), torch.from_numpy(logits))
        ref = _reference(SPEC, experts, shared, bias, x, logits)
        idx, _ = oracle.route(logits, bias, SPEC.k, SPEC.s)
        sent = [int(len(s)) for s in ep.dispatch_plan(torch.from_numpy(idx.astype(np.int64)))]
        out[rank] = (_normwise(y.numpy(), ref.y), np.array_equal(idx, ref.idx),
                     np.array_equal(oracle.permute(idx, SPEC.E)[0], ref.off), sent)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("mode", ["decode", "prefill"])
def test_two_ranks_match_single_rank_oracle_gloo(mode):
    world = 2
    mgr = mp.get_context("spawn").Manager()  # no fork of this (threaded) process
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), mode, out), nprocs=world, join=True)
    for rank in range(world):
        err, idx_ok, off_ok, sent = out[rank]
        assert idx_ok and off_ok
        assert err <= 1e-3, (rank, err)
        assert sum(sent) >= 1
    if mode == "prefill":
        # rows go to both owners (each rank's tokens name experts of both halves)
        assert all(min(out[r][3]) > 0 for r in range(world))
