"""Delayed scaling (amax history ring) on the GPU against the oracle's ring:
codes, the scale each call used, and the ring state after every call, bit for
bit, over a sequence of tensors whose magnitudes rise and fall."""
import numpy as np
import pytest
import torch

import oracle
import scaled_precision_gemm_gb300 as spg
from synthetic_inputs import bf16_bits_to_f32, f32_to_bf16_bits, normal_bf16
from tests.gpu_common import cuda_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("history,shape", [(4, (64, 256)), (16, (1024, 1536)), (1, (3, 40))])
def test_delayed_ring_sequence_matches_oracle(history, shape):
    ring = spg.fp8_scale_ring(history, initial_scale=0.01)
    ref = oracle.DelayedScaleRing(history, initial_scale=0.01)
    for step, mag in enumerate([1.0, 30.0, 0.5, 0.5, 0.0, 2.0, 0.1]):
        x = f32_to_bf16_bits(bf16_bits_to_f32(normal_bf16(shape, seed=step)) * np.float32(mag))
        codes, used = spg.quantize_fp8_tensor_delayed(cuda_bf16(x), ring, history)
        rc, rused = ref.step(x)
        torch.cuda.synchronize()
        assert used[0].item() == float(rused), step
        assert np.array_equal(codes.cpu().numpy(), rc), step
        r = ring.cpu().numpy()
        assert np.array_equal(r[:history], ref.hist), step
        assert r[history] == ref.scale[0], step
        assert r.view(np.uint32)[history + 1] == 0          # per-call amax slot cleared
        assert r.view(np.uint32)[history + 2] == 0          # block counter reset
        assert r.view(np.uint32)[history + 3] == ref.idx[0]
