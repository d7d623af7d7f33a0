"""GPU parity on the expert-sharing decode workloads (batches of 4, 5, 6 and 8 tokens whose
assignments share experts; "b12x" README, DeepSeek V4 Flash MoE benchmark): few experts with
many rows each, down to every token using the same k experts."""
import pytest
import torch

import synth
from test_gpu_moe import moe, run_and_check  # noqa: F401  (fixture + checker)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T", [4, 5, 6, 8])
@pytest.mark.parametrize("share", [0, 40, 80, 100])
def test_sharing_workloads(moe, T, share):  # noqa: F811
    cs = synth.CONFIGS["decode"]
    lg = synth.gen_sharing_logits(cs, T, share, device="cuda")
    run_and_check(moe, cs, T, logits=lg)
