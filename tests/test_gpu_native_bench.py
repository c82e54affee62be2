"""ssv_bench (native timing utility) runs every op of the library on the
named synthetic workloads and reports positive times and work figures."""
import json

import pytest

from diffusion_speculative_verification_gb300 import ssv
from gpu_common import ensure_built

pytestmark = pytest.mark.gpu


def setup_module():
    ensure_built()


@pytest.mark.parametrize("config", ["tiny", "gqa1p7b", "prefill"])
def test_native_bench(config):
    j = json.loads(ssv.bench(config, 2))
    assert j["config"] == config
    for key in ("rope_us", "attn_us", "commit_us"):
        assert j[key][0] > 0, key
    assert j["attn_bytes"] > 0 and j["attn_flops"] > 0
    if config == "prefill":
        assert j["accept_us"][0] == 0 and j["lmhead_us"][0] == 0 and j["commit_bytes"] > 0
    else:
        assert j["accept_us"][0] > 0 and j["lmhead_us"][0] > 0
        assert j["lmhead_flops"] > 0 and j["lmhead_hidden"] == {"tiny": 64, "gqa1p7b": 2048}[config]
