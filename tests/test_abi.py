"""The C-ABI library loads, exports every function include/pm.h declares, and sizes the
KV cache as the audit's section 6 states (no GPU needed)."""
import json
import os
import re

from full_duplex_speech_moshi_gb300 import inputs as I
from full_duplex_speech_moshi_gb300 import pm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions(header="pm.h"):
    src = open(os.path.join(ROOT, "include", header)).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pm_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol():
    L = pm.lib()
    headers = sorted(f for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h"))
    assert headers == ["pm.h", "pm_mimi.h"]
    assert set(declared_functions("pm.h")) == set(pm.EXPORTS)
    assert set(declared_functions("pm_mimi.h")) == set(pm.MIMI_EXPORTS)
    for n in pm.EXPORTS + pm.MIMI_EXPORTS:
        assert hasattr(L, n), n


def test_kv_cache_bytes_matches_page():
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "personaplex_inventory.json")))
    cfg = pm.make_config(I.FULL.asdict(), B_max=1)
    assert pm.pm_kv_cache_bytes(cfg) == g["temporal_kv_bytes_32_layers_bf16_B1"]
    cfg16 = pm.make_config(I.FULL.asdict(), B_max=16)
    assert pm.pm_kv_cache_bytes(cfg16) == 16 * g["temporal_kv_bytes_32_layers_bf16_B1"]


def test_config_struct_layout():
    # the ctypes mirror must match the C struct: 11 ints, 32 delays, 2 ints, 2 floats, 10 ints, flags
    import ctypes as C
    assert C.sizeof(pm.pm_config) == 4 * (11 + 32 + 2 + 2 + 10 + 1)
