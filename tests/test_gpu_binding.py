"""The binding's default stream: with stream=None every call is issued on
torch's current stream.  The fast lookup the binding uses must give the same
handle as torch.cuda.current_stream(), outside and inside a
`torch.cuda.stream` block, and a call issued inside such a block must be
ordered on that stream."""
import numpy as np
import pytest

from hierarchical_quantized_kv_gb300 import qs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    import torch as t
    assert t.cuda.is_available(), "GPU tests need CUDA"
    import __graft_entry__
    __graft_entry__.build()
    return t


def test_default_stream_handle_is_torch_current_stream(torch):
    assert qs._current_stream_handle() == torch.cuda.current_stream().cuda_stream
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        assert qs._current_stream_handle() == side.cuda_stream
        assert qs._current_stream_handle() == torch.cuda.current_stream().cuda_stream
    assert qs._current_stream_handle() == torch.cuda.current_stream().cuda_stream


def test_call_inside_a_stream_block_runs_on_that_stream(torch):
    """qs_state_reset issued on a side stream after a kernel that fills the
    counters on the same stream: the reset must see (and clear) them."""
    cache = qs.Cache(2, 2, 2)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        cache.state.fill_(7)
        qs.qs_state_reset(cache)
    side.synchronize()
    assert int(cache.state.abs().sum().item()) == 0
    assert np.all(qs.qs_get_errors(cache) == 0)
