"""moe_ffn_decode_static (the decode on the library's own per-device scratch,
for callers that cannot allocate device memory) against moe_ffn_decode with a
caller workspace: two consecutive calls on different tokens give the same
bits as the workspace entry point, on the tiny layer and on the full decode
layer. Collected last, so it also runs after every other GPU test in the same
process."""
import numpy as np
import pytest
import torch

import bit_codebook_quantized_dequant_gb300 as M
from bit_codebook_quantized_dequant_gb300 import synth as S
from bit_codebook_quantized_dequant_gb300.workload import Workspace, build_layer, to_dev_u16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny-decode", "decode-b1"])
def test_static_scratch_matches_workspace_decode(name):
    cfg = dict(S.WORKLOADS[name])
    seed = S.workload_seed(name) + 7
    dl = build_layer(seed, 0, cfg)
    ws = Workspace(dl, 0)
    xs = S.tokens(seed, cfg, 2, start=300)
    H = cfg["H"]
    for t in range(2):  # two consecutive calls
        x = to_dev_u16(xs[t])
        y_ref = torch.zeros(H, dtype=torch.float32, device="cuda")
        y = torch.full((H,), float("nan"), dtype=torch.float32, device="cuda")
        st_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        M.moe_ffn_decode(dl.desc(), x, y_ref, ws.ptr, ws.nbytes, st_ref)
        M.moe_ffn_decode_static(dl.desc(), x, y, st)
        torch.cuda.synchronize()
        assert st_ref.item() == 0 and st.item() == 0
        np.testing.assert_array_equal(y.cpu().numpy(), y_ref.cpu().numpy())
