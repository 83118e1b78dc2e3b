"""The Python binding rejects tensors it cannot hand to the library, on the
host and before anything is launched (CPU: no GPU is needed to reach these
checks)."""
import pytest
import torch

import cross_entropy_loss_ce_gb300 as gbce


class FakeCuda:
    """Stands in for a CUDA tensor where only its device is looked at."""

    def __init__(self, index: int):
        self.is_cuda = True
        self.device = torch.device("cuda", index)


class FakeStream:
    def __init__(self, index: int):
        self.device = torch.device("cuda", index)
        self.cuda_stream = 0


def test_one_device_for_all_tensors():
    assert gbce._call_device(("a", FakeCuda(1)), ("b", None), ("c", FakeCuda(1))) == \
        torch.device("cuda", 1)


def test_tensors_on_two_devices_are_rejected():
    with pytest.raises(ValueError, match="targets is on cuda:1"):
        gbce._call_device(("logits", FakeCuda(0)), ("targets", FakeCuda(1)))


def test_a_host_tensor_is_rejected():
    with pytest.raises(ValueError, match="loss must be a CUDA tensor"):
        gbce._call_device(("logits", FakeCuda(0)), ("loss", torch.zeros(())))


def test_a_stream_of_another_device_is_rejected():
    with pytest.raises(ValueError, match="stream is on cuda:1"):
        gbce._stream_handle(FakeStream(1), torch.device("cuda", 0))


def test_wrappers_reject_host_tensors_before_loading_anything():
    x = torch.zeros((2, 3))
    t = torch.zeros((2,), dtype=torch.int64)
    for call in (lambda: gbce.ce_fwd_bwd(x, t), lambda: gbce.softmax_fwd(x, x),
                 lambda: gbce.softmax_bwd(x, x, x), lambda: gbce.ce_fwd_bwd_ex(x, t),
                 lambda: gbce.ce_fwd_bwd_noalloc(x, t), lambda: gbce.scale_rows(x, 1.0)):
        with pytest.raises(ValueError, match="must be a CUDA tensor"):
            call()
