"""The E4M3 bytes the tensor-core GEMM tests feed for the int4 codes -7..7
(written out from the format's definition) equal torch's own float32 ->
float8_e4m3fn conversion on the CPU."""
import numpy as np
import torch

from tests.test_gpu_gemm import e4m3_bytes


def test_e4m3_table_matches_torch_conversion():
    v = np.arange(-7, 8)
    want = torch.tensor(v, dtype=torch.float32).to(torch.float8_e4m3fn)
    want = want.view(torch.uint8).numpy()
    assert np.array_equal(e4m3_bytes(v), want)
    back = torch.from_numpy(e4m3_bytes(v).astype(np.uint8)).view(torch.float8_e4m3fn)
    assert np.array_equal(back.to(torch.float32).numpy(), v.astype(np.float32))
