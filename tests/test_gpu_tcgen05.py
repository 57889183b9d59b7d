"""The tensor-core building blocks (tensor memory, the asynchronous MMA, the
shared-memory descriptors, the tensor-memory load layouts) against a host
product: tq_selftest_tcgen05 computes A . B three ways."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def test_tcgen05_building_blocks():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from online_kv_cache_encode_gb300 import build
    build.build()
    from online_kv_cache_encode_gb300 import tq
    g = torch.Generator().manual_seed(7)
    A = torch.randn(128, 256, generator=g).half()
    B = torch.randn(256, 16, generator=g).half()
    ref = A.double().numpy() @ B.double().numpy()
    st = tq.new_status()
    out = tq.selftest_tcgen05(A.cuda(), B.cuda(), st).cpu().numpy().astype(np.float64)
    torch.cuda.synchronize()
    assert st.item() == 0
    for i, what in enumerate(["A in tensor memory", "fragment-layout read back", "A in shared memory",
                              "A through the fragment-layout store"]):
        np.testing.assert_allclose(out[i], ref, rtol=1e-5, atol=1e-4, err_msg=what)
    # B in the MN-major layout: the descriptor reading the prefill kernel uses
    # (leading byte offset = step between 8-row groups along K, stride byte
    # offset = step between 8-element groups along N, the roles they have in
    # the K-major layout) must match, and the other must not
    match = [bool(np.allclose(out[i], ref, rtol=1e-5, atol=1e-4)) for i in (4, 5)]
    print("MN-major B, readings (K step, N step) = (128, 4096) / (4096, 128):", match)
    assert match == [True, False], match
