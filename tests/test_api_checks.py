"""The torch layer's checks of caller-supplied outputs and workspaces (CPU: the
checks run before any pointer reaches the library, so a wrong tensor raises a
Python error instead of reaching a kernel)."""
import pytest
import torch

from lm_head_kl_fkl_b300 import api

CUDA0 = torch.device("cuda", 0)


@pytest.mark.parametrize("t, dtype, shape, err", [
    (torch.empty(7, dtype=torch.float32), torch.float32, (8,), ValueError),          # lse shorter than N
    (torch.empty(8, dtype=torch.float64), torch.float32, (8,), TypeError),           # wrong dtype
    (torch.empty(2, dtype=torch.float32), torch.float32, (1,), ValueError),          # loss not [1]
    (torch.empty(4, 3, dtype=torch.bfloat16), torch.bfloat16, (4, 4), ValueError),   # dh not [N, d]
    (torch.empty(5, 4, dtype=torch.bfloat16), torch.float32, (5, 4), TypeError),     # dW in bf16
    (torch.empty(8, dtype=torch.float32), torch.float32, (8,), ValueError),          # right shape, host memory
    ("not a tensor", torch.float32, (8,), TypeError),
])
def test_output_checks(t, dtype, shape, err):
    with pytest.raises(err):
        api._expect_out(t, "out", dtype, shape, CUDA0)


def test_workspace_must_be_device_memory():
    with pytest.raises(ValueError, match="CUDA tensor"):
        api._ws_bytes(torch.empty(1024, dtype=torch.uint8), CUDA0)
    with pytest.raises(TypeError):
        api._ws_bytes(bytearray(1024), CUDA0)


def test_grad_scalar_checks():
    assert api._grad_scalar(None, CUDA0) is None
    with pytest.raises(ValueError, match="one-element"):
        api._grad_scalar(torch.ones(2), CUDA0)
    with pytest.raises(TypeError):
        api._grad_scalar(torch.ones(1, dtype=torch.float64), CUDA0)
    with pytest.raises(ValueError, match="CUDA tensor"):
        api._grad_scalar(torch.ones(1), CUDA0)
