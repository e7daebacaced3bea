"""sigma-routed sequence sharding with the GPU kernels: every rank's local
problem (from the library's routing plan) runs through sa_forward on one GPU,
one rank after another, and the reassembled output is checked against the
fp64 oracle and against the whole sequence run at once.  (The exchanges
themselves are covered on gloo ranks in test_shard.py; one GPU per box here.)
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import stochastic_sliding_window_gb300 as sa
from gpu_helpers import Inputs, compare, gather_rows, perms, sample_rows
from stochastic_sliding_window_gb300 import shard

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("world", [2, 4, 8])
@pytest.mark.parametrize("w,causal", [(128, True), (64, False)])
def test_sharded_long_prefill_matches_whole_sequence(world, w, causal):
    n = 32768
    inp = Inputs(1, n, 32, 8, 128, seed=21 + world, gates=False)
    perm, perm_d = perms(9, world, 1, n)
    whole = sa.sa_forward(inp.q, inp.k, inp.v, perm_d, w, causal=causal)
    out = torch.empty_like(whole)
    for p in shard.plans(perm[0].astype(np.int32), w, world):
        t = torch.from_numpy(p.tokens.astype(np.int64)).cuda()
        lp = torch.from_numpy(p.local_perm[None].copy()).cuda()
        y = sa.sa_forward(inp.q[:, t].contiguous(), inp.k[:, t].contiguous(),
                          inp.v[:, t].contiguous(), lp, w, causal=causal)
        own = torch.from_numpy(p.own_local.astype(np.int64)).cuda()
        out[0, torch.from_numpy(p.own_tokens.astype(np.int64)).cuda()] = y[0, own]
    rows = sample_rows(1, n, 200, seed=world)
    want = oracle.sa_rows(inp.case.q, inp.case.k, inp.case.v, perm, w, causal, rows=rows)
    compare(gather_rows(out, rows), want, f"sharded over {world}")
    assert (out.float() - whole.float()).abs().max().item() <= 2e-2
