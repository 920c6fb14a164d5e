"""moe_stream_read, the benchmark's size-matched read ceiling: it must read every byte it is given
once. Its XOR fold of the buffer's 32-bit words is compared with numpy's fold of the same bytes
(one grid stride, several strides with a ragged tail, a single 16-byte word)."""
import numpy as np
import pytest
import torch

from moe_expert_ffn_histogram_gb300 import capi

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.mark.parametrize("nbytes", [16, 4096, (1 << 20) + 48, (64 << 20) + 16])
def test_stream_read_folds_every_word(nbytes):
    g = torch.Generator(device="cpu").manual_seed(nbytes % 9973)
    host = torch.randint(0, 256, (nbytes + 64,), dtype=torch.uint8, generator=g)
    buf = host.to(DEV)
    sink = torch.zeros(1, dtype=torch.int32, device=DEV)
    capi.stream_read(buf, nbytes, sink)
    torch.cuda.synchronize()
    want = int(np.bitwise_xor.reduce(host[:nbytes].numpy().view(np.uint32)))
    assert int(sink.item()) & 0xFFFFFFFF == want
    # the sink is not cleared: folding the same bytes into it again brings it back to zero
    capi.stream_read(buf, nbytes, sink)
    torch.cuda.synchronize()
    assert int(sink.item()) == 0


def test_stream_read_binding_checks():
    buf = torch.zeros(1024, dtype=torch.uint8, device=DEV)
    sink = torch.zeros(1, dtype=torch.int32, device=DEV)
    with pytest.raises(capi.MoeError):
        capi.stream_read(buf, 1000, sink)          # not a multiple of 16
    with pytest.raises(ValueError):
        capi.stream_read(buf, 2048, sink)          # past the buffer
