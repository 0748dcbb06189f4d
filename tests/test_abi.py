"""Host-side checks of the C ABI: the library builds, loads without a GPU,
exports every function the headers declare, and rejects bad configurations
before touching the device."""
import ctypes
import os
import re
import shutil

import pytest

from text_embedding_encoder_gb300 import binding, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(tee_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def built_lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("no CUDA toolkit")
    from text_embedding_encoder_gb300 import build
    path = build.build()
    return binding.load(path)


def test_headers_declare_the_boundary():
    names = _declared_functions()
    for required in ("tee_create", "tee_load_weights", "tee_encode", "tee_encode_device", "tee_destroy",
                     "tee_last_error"):
        assert required in names
    assert names == set(binding.SIGNATURES), names ^ set(binding.SIGNATURES)


def test_library_exports_every_declared_symbol(built_lib):
    for name in _declared_functions():
        assert hasattr(built_lib, name), name


def _cfg(**over):
    c = binding.config_from_shape(synth.TINY, "fp32", 512, 8)
    for k, v in over.items():
        setattr(c, k, v)
    return c


@pytest.mark.parametrize("field,value", [
    ("head_dim", 32), ("hidden", 200), ("n_layers", 0), ("intermediate", 100), ("dtype", 7),
    ("max_tokens", 0), ("max_texts", 0), ("global_every", 0), ("window", -1), ("vocab", 0),
    ("emb_norm", 2), ("final_norm", -1), ("proj_dim", 100), ("proj_dim", 2048), ("proj_dim", -128),
])
def test_create_rejects_bad_config_without_a_device(built_lib, field, value):
    ctx = ctypes.c_void_p(123)
    cfg = _cfg(**{field: value})
    rc = built_lib.tee_create(ctypes.byref(cfg), 0, ctypes.byref(ctx))
    assert rc == binding.TEE_EINVAL
    assert ctx.value is None
    assert built_lib.tee_last_error(None).decode() != ""


def test_null_safety_without_a_device(built_lib):
    built_lib.tee_destroy(None)
    assert built_lib.tee_encode(None, None, None, 1, None) == binding.TEE_EINVAL
    assert built_lib.tee_encode_tokens(None, None, None, 1, None) == binding.TEE_EINVAL
    assert built_lib.tee_encode_tokens_device(None, None, None, None, 1, None, None) == binding.TEE_EINVAL
    assert built_lib.tee_create(None, 0, None) == binding.TEE_EINVAL
