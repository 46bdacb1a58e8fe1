"""mk_decode_step_static: the decode step with its counters in the fixed
device array gives the same logits as mk_decode_step, call after call, and
allocates no device memory.  Collected last on purpose (file name), so it also
runs after every other GPU test in the same process."""
from __future__ import annotations

import ctypes as C

import numpy as np
import pytest
import torch

from persistent_moe_decode_gb300 import mk
from persistent_moe_decode_gb300.configs import TINY, WORKLOADS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from persistent_moe_decode_gb300 import build
    build.build()


@pytest.mark.parametrize("name", ["tiny", "mid_8k"])
def test_static_counter_step_matches_the_regular_step_twice_in_a_row(name):
    from persistent_moe_decode_gb300.runner import StepRunner
    run = StepRunner(WORKLOADS[name], device="cuda")
    try:
        run.schedule()
        run.launch()
        torch.cuda.synchronize()
        run.check_status()
        ref = run.logits.clone()
        idx_ref, w_ref = run.dec.routing()
        for call in range(2):
            run.logits.fill_(float("nan"))
            torch.cuda.synchronize()
            free_before = torch.cuda.mem_get_info()[0]
            run.dec.decode_static(run.logits)
            torch.cuda.synchronize()
            free_after = torch.cuda.mem_get_info()[0]
            run.check_status()
            assert torch.equal(run.logits, ref), f"call {call}"
            idx, w = run.dec.routing()
            assert np.array_equal(idx, idx_ref) and np.array_equal(w, w_ref)
            if call == 1:   # the first call may load the module; later ones allocate nothing
                assert free_after == free_before
        # and the regular entry point still agrees afterwards
        run.launch()
        torch.cuda.synchronize()
        run.check_status()
        assert torch.equal(run.logits, ref)
    finally:
        run.close()


def test_static_counter_step_rejects_handles_beyond_the_array():
    """A model deep enough to need more counter words than the array holds is
    refused before anything runs (every layer reuses the same weight tensors)."""
    from persistent_moe_decode_gb300.synth import make_kv_pools, make_model
    import dataclasses
    one = dataclasses.replace(TINY, n_layers=1)
    model = make_model(one, 7, torch.device("cuda"))
    kp, vp = make_kv_pools(one, 8, 1.0, 7, torch.device("cuda"))
    L = 2100   # 32 + 2100 * 32 words > 65536
    cfg = mk.make_config(dataclasses.replace(TINY, n_layers=L), 16, 4, 8)
    keep = []

    def arr(t):
        a = (C.c_void_p * L)(*([t[0].data_ptr()] * L))
        keep.append(a)
        return C.cast(a, C.POINTER(C.c_void_p))

    w = mk.mk_weights(embed=model.embed.data_ptr(), lm_head=model.lm_head.data_ptr(),
                      final_norm=model.final_norm.data_ptr(), attn_norm=arr(model.attn_norm),
                      w_qkv=arr(model.w_qkv), w_o=arr(model.w_o), w_router=arr(model.w_router),
                      w_gate=arr(model.w_gate), w_up=arr(model.w_up), w_down=arr(model.w_down),
                      k_pool=arr(kp), v_pool=arr(vp))
    h = mk.mk_create(cfg, w)
    try:
        logits = torch.empty(1, TINY.vocab, device="cuda")
        rc = mk.lib().mk_decode_step_static(h, C.c_void_p(logits.data_ptr()), None)
        assert rc == mk.MK_ERR_BAD_CONFIG
    finally:
        mk.mk_destroy(h)
