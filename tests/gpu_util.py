"""Helpers shared by the GPU parity tests (inputs on the host for the oracle)."""
import numpy as np
import pytest
import torch

import oracle


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def host(t: torch.Tensor) -> np.ndarray:
    """A device or host fp32/bf16 tensor (2-D, unit column stride) as an oracle input."""
    return oracle.host_array(t.detach().to("cpu"))


def oracle_ce(logits_host: torch.Tensor, targets_host: torch.Tensor, rows=None,
              want_grad=True, ignore_index=-100):
    """Oracle result for the listed rows plus the batch-wide n and mean loss."""
    V = logits_host.shape[1]
    x = oracle.host_array(logits_host)
    t = targets_host.numpy()
    n, bad = oracle.ce_count(t, V, ignore_index)
    grad, row_loss = oracle.ce_rows(x, t, V, n, ignore_index, rows=rows, want_grad=want_grad)
    return dict(grad=grad, row_loss=row_loss, n=n, bad=bad)
