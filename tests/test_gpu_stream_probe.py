"""The streaming reference kernel behind bench.py's `stream_ref` figures (te_stream_probe): it must
move exactly the bytes it is said to move, so that its time is a fair floor for a kernel with the
same traffic.  Each written 16-byte vector is the exclusive or of the `ratio` vectors read before
it; read-only mode writes nothing."""

import numpy as np
import pytest
import torch

import fp8_transformer_gb300 as te
from parity import Guarded

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("ratio", [1, 2, 4])
@pytest.mark.parametrize("n_out", [1, 1000, 300001])
def test_stream_probe_moves_the_stated_bytes(ratio, n_out):
    g = torch.Generator(device="cuda").manual_seed(ratio * 7 + n_out)
    src = torch.randint(0, 2 ** 31 - 1, (n_out * ratio * 4,), generator=g, dtype=torch.int32,
                        device="cuda")
    dst = Guarded((n_out * 4,), torch.int32)
    te.stream_probe(src, dst.t, write_bytes=n_out * 16, ratio=ratio)
    dst.check("stream probe output")
    want = np.bitwise_xor.reduce(src.cpu().numpy().reshape(n_out, ratio, 4), axis=1).reshape(-1)
    assert np.array_equal(dst.t.cpu().numpy(), want)


def test_stream_probe_read_only_writes_nothing():
    src = torch.ones(1 << 20, dtype=torch.int32, device="cuda")
    dst = Guarded((16,), torch.int32)
    before = dst.t.clone()
    te.stream_probe(src, dst.t, write_bytes=0, read_only_bytes=src.numel() * 4)
    dst.check("read-only probe")
    assert torch.equal(dst.t, before)
