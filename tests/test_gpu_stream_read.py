"""The read-floor reference (ssv_stream_read): every 32-bit word of the buffer
is read once -- its XOR checksum equals the one numpy forms -- for sizes that
leave CTAs with empty, partial and full ranges."""
import numpy as np
import pytest
import torch

from diffusion_speculative_verification_gb300 import ssv
from gpu_common import ensure_built

pytestmark = pytest.mark.gpu


def setup_module():
    ensure_built()


@pytest.mark.parametrize("nbytes", [16, 4096, 65536 + 48, 5 << 20, (64 << 20) + 16])
def test_stream_read_checksum(nbytes):
    rng = np.random.default_rng(nbytes)
    words = rng.integers(0, 1 << 32, size=nbytes // 4, dtype=np.uint64).astype(np.uint32)
    buf = torch.from_numpy(words.view(np.int32)).cuda()
    out = torch.zeros(1, dtype=torch.int32, device="cuda")
    ssv.stream_read(buf, out)
    torch.cuda.synchronize()
    want = np.bitwise_xor.reduce(words)
    assert int(out.cpu().numpy().view(np.uint32)[0]) == int(want)
