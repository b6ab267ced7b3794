"""The streaming calibration (ckv_calibrate_stream): the decode's data movement
with no compute runs to completion on a packed cache, with and without the
split rendezvous, raises no device flag and leaves its counters at zero."""
import pytest

torch = pytest.importorskip("torch")

import compressed_kv_attention_gb300 as ckv  # noqa: E402
from compressed_kv_attention_gb300 import inputs  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("rendezvous", [False, True])
def test_calibrate_stream_runs_clean(rendezvous):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    D, Hkv, T = 512, 2, 4096
    cache = ckv.PackedCache(D, Hkv, 1, T, inputs.tbq_signs(D), device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    rec = 23 * D + 32
    for n_split in (1, 7, 64):
        for _ in range(3):
            ckv.calibrate_stream(cache.data, T // 16, rec, Hkv, n_split, rendezvous, ws)
    torch.cuda.synchronize()
    assert ckv.read_device_flag(ws) == 0
    assert torch.all(ws[64:] == 0)


def test_calibrate_stream_rejects_bad_arguments():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    buf = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(ckv.CkvError):
        ckv.calibrate_stream(buf, 16, 100, 1, 1, False, ws)      # record not a multiple of 16
    with pytest.raises(ckv.CkvError):
        ckv.calibrate_stream(buf, 16, 16384, 1, 1, False, ws)    # 16 records of 16 KB exceed the ring
    with pytest.raises(ckv.CkvError):
        ckv.calibrate_stream(buf, 16, 1024, 4, 1024, True, ws)  # rendezvous grid cannot fit at once
