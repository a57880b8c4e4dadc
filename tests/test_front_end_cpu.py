"""Host-side checks of the autograd front end (chunk_loss.py): a negative
chunk size and an unknown reduction are refused before anything reaches the
library, mirroring the plugin's validation of a non-positive chunk size."""
import pytest
import torch

from lm_head_linear_chunked_gb300.chunk_loss import ChunkLoss, linear_cross_entropy


def _head():
    return torch.nn.Linear(16, 32, bias=False, dtype=torch.bfloat16)


def test_chunk_loss_rejects_negative_chunk_rows():
    with pytest.raises(ValueError):
        ChunkLoss(_head(), chunk_rows=-1)


def test_chunk_loss_rejects_unknown_reduction():
    with pytest.raises(ValueError):
        ChunkLoss(_head(), reduction="avg")


def test_chunk_loss_keeps_its_settings():
    head = _head()
    m = ChunkLoss(head, chunk_rows=128, ignore_index=-1, reduction="sum")
    assert m.head is head and m.chunk_rows == 128 and m.ignore_index == -1 and m.reduction == "sum"


@pytest.mark.parametrize("kw", [{"chunk_rows": -5}, {"reduction": "none"}])
def test_linear_cross_entropy_rejects_bad_arguments(kw):
    X = torch.zeros(4, 16, dtype=torch.bfloat16)
    W = torch.zeros(32, 16, dtype=torch.bfloat16)
    y = torch.zeros(4, dtype=torch.int64)
    with pytest.raises(ValueError):
        linear_cross_entropy(X, W, y, **kw)
