"""The allocation-free pooling entry point, tee_pool_l2_noalloc.

It serves callers that cannot allocate device memory (a host framework that
owns every device byte through its own pool, or a latency-critical path that
cannot take an allocation's implicit synchronisation), so it keeps its scratch
in fixed-size device arrays of the library instead of a context's workspace.
This test calls it through the C ABI twice in a row, with different inputs,
and checks each result against the oracle's pooling (the per-text mean scaled
to unit length, in fp64) and against the context-based tee_op_pool_l2, within
the tolerance the pool step test uses.  It runs last (file name) so a failure
here cannot hide failures elsewhere, and it needs nothing from earlier tests.
"""
import numpy as np
import pytest

import oracle
from text_embedding_encoder_gb300 import binding, synth

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

POOL_ATOL = 2e-6


def _noalloc(lib, x, d_cu, cu, n, H, out):
    return lib.tee_pool_l2_noalloc(x.data_ptr(), d_cu.data_ptr(), cu.ctypes.data, n, H, out.data_ptr(), 0)


def test_pool_noalloc_matches_oracle_and_pool_op(lib):
    shape = synth.TINY
    H = shape.hidden
    enc = binding.Encoder(shape, "fp32", max_tokens=4096, max_texts=64)   # only for the context entry point
    rng = np.random.default_rng(17)
    for lengths in ([1, 63, 64, 65, 300, 2, 129], [1000, 7, 128, 1, 2000]):
        ids, cu = synth.make_batch(lengths, shape.vocab, seed=len(lengths))
        T, n = int(cu[-1]), len(lengths)
        x_h = rng.standard_normal((T, H)).astype(np.float32)
        x = torch.from_numpy(x_h).cuda()
        d_cu = torch.from_numpy(cu).cuda()
        ref = torch.empty(n, H, device="cuda")
        got = torch.full((n, H), float("nan"), device="cuda")
        enc.op("tee_op_pool_l2", x, d_cu, cu, n, ref, 0)
        rc = _noalloc(lib, x, d_cu, cu, n, H, got)
        assert rc == binding.TEE_OK, lib.tee_last_error(None).decode()
        torch.cuda.synchronize()
        got_h = got.cpu().numpy().astype(np.float64)
        want = np.stack([oracle.pool_l2(x_h[cu[j]:cu[j + 1]]) for j in range(n)])
        np.testing.assert_allclose(got_h, want, atol=POOL_ATOL, rtol=0)
        np.testing.assert_allclose(got_h, ref.cpu().numpy(), atol=POOL_ATOL, rtol=0)
        np.testing.assert_allclose(np.linalg.norm(got_h, axis=1), 1.0, atol=1e-5)
    enc.close()


def test_pool_noalloc_rejects_oversized_input(lib):
    n = 9000                                                  # more texts than the scratch holds
    cu = np.arange(n + 1, dtype=np.int32)
    x = torch.zeros(n, 256, device="cuda")
    d_cu = torch.from_numpy(cu).cuda()
    out = torch.empty(n, 256, device="cuda")
    rc = _noalloc(lib, x, d_cu, cu, n, 256, out)
    assert rc == binding.TEE_ETOOLONG
    assert "TEE_POOL_NOALLOC_MAX_TEXTS" in lib.tee_last_error(None).decode()


def test_pool_noalloc_rejects_misaligned_buffers(lib):
    """A view that starts one float into its storage is refused before any
    launch (the kernels move rows as 16-byte vectors)."""
    H = 256
    cu = np.array([0, 3, 8], dtype=np.int32)
    x = torch.zeros(9, H, device="cuda")
    d_cu = torch.from_numpy(cu).cuda()
    out = torch.zeros(3 * H + 1, device="cuda")
    x_bad = x.view(-1)[1:]
    rc = lib.tee_pool_l2_noalloc(x_bad.data_ptr(), d_cu.data_ptr(), cu.ctypes.data, 2, H,
                                 out.data_ptr(), 0)
    assert rc == binding.TEE_EINVAL
    assert "16-byte" in lib.tee_last_error(None).decode()
    rc = lib.tee_pool_l2_noalloc(x.data_ptr(), d_cu.data_ptr(), cu.ctypes.data, 2, H,
                                 out[1:].data_ptr(), 0)
    assert rc == binding.TEE_EINVAL
    torch.cuda.synchronize()
    assert float(out.abs().sum()) == 0.0                      # nothing was written
