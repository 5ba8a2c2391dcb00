"""moe_route_noalloc: routing for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc (their device memory belongs to another
allocator or runtime, or they are plain C code without a device allocator),
so libmoe offers one routing entry point that takes no workspace and uses a
fixed scratch array inside the library instead.  This test calls it through
the C ABI twice in a row, on different inputs, and checks each call against
moe_route (which uses a caller workspace) on the same inputs.  It runs last
so that a failure here does not stop the other GPU tests, and it passes both
alone in a fresh process and after the rest of the suite.
"""

import numpy as np
import pytest
import torch

import synth_inputs as si

pytestmark = pytest.mark.gpu


def _outputs(sh, device):
    T, E, k = sh.T, sh.E, sh.top_k
    return {
        "logits": torch.empty(T, E, dtype=torch.float32, device=device),
        "topk_idx": torch.empty(T, k, dtype=torch.int32, device=device),
        "topk_w": torch.empty(T, k, dtype=torch.float32, device=device),
        "counts": torch.empty(E, dtype=torch.int32, device=device),
        "offsets": torch.empty(E + 1, dtype=torch.int32, device=device),
        "perm_token": torch.empty(T * k, dtype=torch.int32, device=device),
        "slot_row": torch.empty(T, k, dtype=torch.int32, device=device),
    }


def test_route_noalloc_matches_route_on_two_calls_in_a_row():
    from mixture_experts_layer_17_gb300 import libmoe
    dev = torch.device("cuda")
    for call, (T, E, k, seed, skew) in enumerate([(3000, 128, 8, 41, False),
                                                  (517, 32, 4, 42, True)]):
        sh = si.custom_shape(T, 512, 256, E, k, seed=seed, skew=skew)
        inp = si.make_inputs(sh, dev, with_grad=False, with_weights=False)
        cfg = libmoe.make_config(sh.T, sh.H, sh.F, sh.E, sh.top_k)
        # reference: moe_route with a caller-owned workspace
        fwd_ws, _, _ = libmoe.moe_workspace_size(cfg)
        ws = torch.empty(fwd_ws, dtype=torch.uint8, device=dev)
        ref = _outputs(sh, dev)
        libmoe.moe_route(cfg, inp["x"], inp["W_r"], inp["logit_bias"], ref["logits"],
                         ref["topk_idx"], ref["topk_w"], ref["counts"], ref["offsets"],
                         ref["perm_token"], ref["slot_row"], ws)
        # the same routing without a workspace (outputs pre-filled with garbage)
        got = {name: torch.full_like(t, -7) for name, t in ref.items()}
        status = torch.full((1,), -1, dtype=torch.int32, device=dev)
        libmoe.moe_route_noalloc(cfg, inp["x"], inp["W_r"], inp["logit_bias"], got["logits"],
                                 got["topk_idx"], got["topk_w"], got["counts"], got["offsets"],
                                 got["perm_token"], got["slot_row"], status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"call {call}: device status {int(status.item())}"
        for name in ("topk_idx", "counts", "offsets", "perm_token", "slot_row"):
            assert torch.equal(got[name], ref[name]), f"call {call}: {name}"
        for name in ("logits", "topk_w"):
            np.testing.assert_allclose(got[name].cpu().numpy(), ref[name].cpu().numpy(),
                                       rtol=1e-6, atol=0, err_msg=f"call {call}: {name}")


def test_route_noalloc_rejects_configurations_beyond_its_scratch():
    from mixture_experts_layer_17_gb300 import libmoe
    # about 104 bytes of scratch per token at top_k = 8 (at most 69,904 tokens fit in
    # 8 MiB at this shape): 200k tokens are rejected
    cfg = libmoe.make_config(200_000, 4096, 1536, 128, 8)
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")   # never read: rejected first
    outs = [torch.zeros(16, dtype=torch.int32, device="cuda") for _ in range(8)]
    with pytest.raises(libmoe.MoeError) as err:
        libmoe.moe_route_noalloc(cfg, x, x, None, None, outs[0], outs[1].float(), outs[2],
                                 outs[3], outs[4], outs[5], None)
    assert err.value.code == 3          # MOE_ERR_WORKSPACE_TOO_SMALL
