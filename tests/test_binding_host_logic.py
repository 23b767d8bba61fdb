"""The binding's argument checks that run before any CUDA call (CPU only):
a call on device tensors refuses host output tensors and a residual that is
not on x's device (its kernels would be handed host pointers, or the in-place
update would land in a staged copy)."""
import pytest
import torch

nv = pytest.importorskip("nvfp4_block_quantization_quantize_gb300")


def test_device_call_refuses_host_outputs():
    with pytest.raises(ValueError):
        nv._out_buf((4, 8), torch.uint8, torch.empty((4, 8), dtype=torch.uint8), torch.device("cuda", 0), False)


def test_device_call_refuses_foreign_residual():
    with pytest.raises(ValueError):
        nv._dev_residual(torch.zeros((4, 16)), torch.device("cuda", 0))
    assert nv._dev_residual(None, torch.device("cuda", 0)) is None
