"""The device copy of the input generator reproduces the host generator's bits."""
import numpy as np
import pytest
import torch

import synth
from synth import device as synth_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,n_tok", [("tiny_8k_g4_d64", 8192), ("gqa40x8_256k", 4096 + 77)])
def test_device_pool_matches_host_pool(name, n_tok):
    w = synth.WORKLOADS[name].with_(n_tok=n_tok)
    bt = synth.block_table(w)
    k_h, v_h = synth.kv_pool(w, 1, bt)
    k_d = torch.zeros(k_h.shape, dtype=torch.int16, device="cuda")
    v_d = torch.zeros_like(k_d)
    synth_dev.fill_kv_pool(w, 1, torch.from_numpy(bt).cuda(), k_d, v_d)
    torch.cuda.synchronize()
    assert np.array_equal(k_d.cpu().numpy().view(np.uint16), k_h)
    assert np.array_equal(v_d.cpu().numpy().view(np.uint16), v_h)
