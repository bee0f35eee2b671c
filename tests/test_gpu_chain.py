"""GPU parity of the chained multi-layer decode: L decode calls per step, built
as ``sparse_mla_decode_gb300.chain`` builds them (each layer one of the pages'
latency workloads, its rows renumbered into a shared pool), captured in one
CUDA graph with programmatic dependent launch on, replayed, and every layer's
output and LSE checked against the oracle's emulated datapath and its fp64
definition."""

import os

import numpy as np
import pytest
import torch

from sparse_mla_decode_gb300 import chain, smla
from tests.gpu_helpers import compare

pytestmark = pytest.mark.gpu


def _poison(sets):
    for calls in sets:
        for c in calls:
            c["out"].fill_(float("nan"))
            c["lse"].fill_(float("nan"))


@pytest.mark.parametrize("shape", ["verify", "tiny"])
def test_graph_captured_layer_chain_matches_the_oracle(shape):
    assert os.environ.get("SMLA_PDL", "1") != "0", "the chain is checked with dependent launch on"
    dev = torch.device("cuda", 0)
    layers, sets_count, steps = 8, 2, 5  # steps rotate over the sets, so outputs are rewritten in the graph
    pool, sets = chain.make_sets(shape, layers, sets_count, dev)
    chain.run_layers(sets[0])  # first calls outside the capture (kernel attributes, tensor-map encoder)
    torch.cuda.synchronize()
    _poison(sets)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(steps):
            chain.run_layers(sets[i % sets_count])
    graph.replay()
    torch.cuda.synchronize()
    assert smla.smla_device_error() == 0
    first = [[c["out"].view(torch.int16).clone() for c in calls] for calls in sets]
    graph.replay()
    torch.cuda.synchronize()
    assert smla.smla_device_error() == 0
    pool_np = pool.cpu().numpy()
    for r, calls in enumerate(sets):
        for l, c in enumerate(calls):
            assert torch.equal(c["out"].view(torch.int16), first[r][l]), f"set {r} layer {l}: replays differ"
            w = dict(c["w"], pools=[pool_np], name=f"{shape} set {r} layer {l}")
            out = c["out"]
            compare(w, out.float().cpu().numpy(), out.view(torch.int16).cpu().numpy().view(np.uint16),
                    c["lse"].cpu().numpy())
