"""The bandwidth probe (lmho_probe_read) reads every byte it is given: its
per-segment XOR of 32-bit words matches one computed on the host."""
import numpy as np
import pytest
import torch

import gen

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nseg,seg_bytes", [(1, 16), (3, 8192), (1001, 16384), (5, 65536), (7, 48)])
def test_probe_read_covers_every_word(gpu_lib, nseg, seg_bytes):
    words = gen.targets(31, 0, (nseg * seg_bytes // 4,), 2 ** 32).astype(np.uint32)
    got = gpu_lib.probe_read(torch.from_numpy(words.view(np.int32)).cuda(), seg_bytes).cpu().numpy().view(np.uint32)
    want = np.bitwise_xor.reduce(words.reshape(nseg, -1), axis=1)
    np.testing.assert_array_equal(got, want)
