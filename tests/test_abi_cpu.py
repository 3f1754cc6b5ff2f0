"""Host-side checks of the C ABI and of the tile layouts (no GPU needed).

* libkvq.so builds, loads, and exports every function include/kvq.h declares;
* the pure host entry points answer (tile sizes, status strings, version);
* the ctypes structs match the C struct sizes;
* every tile layout is a bijection onto its tile bytes, and the decode
  kernel's per-lane 16-byte reads are contiguous and bank-conflict free.
"""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kvq.h")


@pytest.fixture(scope="module")
def lib():
    from quantized_kv_cache_kvq_gb300 import build as b

    b.build()
    import quantized_kv_cache_kvq_gb300 as kvq

    return kvq.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s+(kvq_[a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert {"kvq_append", "kvq_decode_attn", "kvq_meter", "kvq_decode_workspace_size"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_host_entry_points(lib):
    import quantized_kv_cache_kvq_gb300 as kvq

    assert lib.kvq_version() == 1
    assert kvq.status_string(0) == "KVQ_OK"
    assert kvq.status_string(8) == "KVQ_ERR_TIMEOUT"
    assert kvq.tile_bytes("bf16", 0) == 4096 and kvq.tile_bytes("e4m3", 0) == 2048
    assert kvq.tile_bytes("int8", 1) == 2048 and kvq.tile_bytes("bf16", 1) == 4096
    assert kvq.tile_bytes("int8", 2) == 32 and kvq.tile_bytes("bf16", 2) == 0
    assert kvq.tile_bytes("e4m3s", 3) == 32 and kvq.tile_bytes("e4m3", 4) == 512
    # INT8 with 32-channel scale groups: 8-bit tiles, 4 fp16 scales per token, no key outlier tile
    assert kvq.tile_bytes("int8g32", 0) == 2048 and kvq.tile_bytes("int8g32", 1) == 2048
    assert kvq.tile_bytes("int8g32", 2) == 128 and kvq.tile_bytes("int8g32", 3) == 128
    assert kvq.tile_bytes("int8g32", 6) == 0 and kvq.tile_bytes("int8g32", 7) == 0


def test_struct_sizes_match_c():
    import quantized_kv_cache_kvq_gb300 as kvq

    assert ctypes.sizeof(kvq._Cache) == 6 * 4 + 8 + 6 * 8 + 8 + 2 * 4 + 8
    assert ctypes.sizeof(kvq.MeterParams) == 32
    lib = kvq.load()
    assert lib.kvq_sizeof(0) == ctypes.sizeof(kvq._Cache)  # as the C compiler laid them out
    assert lib.kvq_sizeof(1) == ctypes.sizeof(kvq.MeterParams)
    assert kvq.MeterParams.delta_req.offset == 16


def test_invalid_arguments_rejected_on_host(lib):
    import quantized_kv_cache_kvq_gb300 as kvq

    # a NULL cache and a bad format are argument errors detected before any device work
    assert lib.kvq_append(None, None, None, 0, None, 1, None, None) == 1
    c = kvq._Cache(9, 0, 8, 1, 0, 0, 0, 16, 16, None, None, 16)
    assert lib.kvq_append(ctypes.byref(c), 16, 16, 0, 16, 1, None, None) == 2
    assert lib.kvq_decode_workspace_size(1, 3, 8) == 0  # 8 % 3 != 0


@pytest.mark.parametrize("plane,fmt,nbytes,elem", [
    ("k", "bf16", 4096, 2), ("k", "e4m3", 2048, 1), ("v", "bf16", 4096, 2), ("v", "e4m3", 2048, 1)])
def test_layouts_are_bijections(plane, fmt, nbytes, elem):
    from quantized_kv_cache_kvq_gb300 import layout as L

    offs = (L.k_offsets if plane == "k" else L.v_offsets)(fmt)
    assert offs.shape == (16, 128)
    assert np.all(offs % elem == 0)
    assert sorted((offs // elem).ravel().tolist()) == list(range(nbytes // elem))


def test_witness_and_scale_layouts_are_bijections():
    from quantized_kv_cache_kvq_gb300 import layout as L

    assert sorted((L.w_offsets() // 2).ravel().tolist()) == list(range(256))
    assert sorted((L.s_offsets() // 2).tolist()) == list(range(16))


def _bank_conflict_free(chunk_idx):
    """32 lanes read 16-byte chunks; the hardware serves 8 lanes per phase: the 8 chunks of a phase
    must fall into 8 distinct 16-byte bank groups (chunk index mod 8)."""
    for ph in range(4):
        grp = [c % 8 for c in chunk_idx[8 * ph:8 * ph + 8]]
        if len(set(grp)) != 8:
            return False
    return True


def test_decode_fragment_reads_are_contiguous_and_conflict_free():
    from quantized_kv_cache_kvq_gb300 import layout as L

    lanes = np.arange(32)
    g, c = lanes >> 2, lanes & 3
    # K 16-bit: read (nt, j) gives lane (g, c) token 8nt+g, channels 32j+8c .. +7
    ko = L.k_offsets("bf16")
    for nt in range(2):
        for j in range(4):
            starts = [ko[8 * nt + gg, 32 * j + 8 * cc] for gg, cc in zip(g, c)]
            assert all(ko[8 * nt + gg, 32 * j + 8 * cc + e] == s + 2 * e for gg, cc, s in zip(g, c, starts) for e in range(8))
            assert starts == [((nt * 4 + j) * 32 + L_) * 16 for L_ in lanes]
            assert _bank_conflict_free([s // 16 for s in starts])
    # K 8-bit: read (nt, jj): token 8nt+g, channels 64jj+16c .. +15
    ko8 = L.k_offsets("e4m3")
    for nt in range(2):
        for jj in range(2):
            starts = [ko8[8 * nt + gg, 64 * jj + 16 * cc] for gg, cc in zip(g, c)]
            assert starts == [((nt * 2 + jj) * 32 + L_) * 16 for L_ in lanes]
            assert all(ko8[8 * nt + gg, 64 * jj + 16 * cc + e] == s + e for gg, cc, s in zip(g, c, starts) for e in range(16))
    # V 8-bit: read mm gives lane (g, c) the A fragments of V^T for channel blocks 2mm and 2mm+1:
    # per block, tokens (2c, 2c+1) then (2c+8, 2c+9), each at channel g then g + 8
    vo = L.v_offsets("e4m3")
    for mm in range(4):
        for half in range(2):
            mt = 2 * mm + half
            for gg, cc, L_ in zip(g, c, lanes):
                base = (mm * 32 + L_) * 16 + 8 * half
                order = [(2 * cc, 16 * mt + gg), (2 * cc + 1, 16 * mt + gg), (2 * cc, 16 * mt + gg + 8),
                         (2 * cc + 1, 16 * mt + gg + 8), (2 * cc + 8, 16 * mt + gg), (2 * cc + 9, 16 * mt + gg),
                         (2 * cc + 8, 16 * mt + gg + 8), (2 * cc + 9, 16 * mt + gg + 8)]
                assert [vo[t, ch] for t, ch in order] == [base + i for i in range(8)]
    # V 16-bit: read mt gives the same eight values of channel block mt as 16-bit elements
    vo16 = L.v_offsets("bf16")
    for mt in range(8):
        for gg, cc, L_ in zip(g, c, lanes):
            base = (mt * 32 + L_) * 16
            order = [(2 * cc, 16 * mt + gg), (2 * cc + 1, 16 * mt + gg), (2 * cc, 16 * mt + gg + 8),
                     (2 * cc + 1, 16 * mt + gg + 8), (2 * cc + 8, 16 * mt + gg), (2 * cc + 9, 16 * mt + gg),
                     (2 * cc + 8, 16 * mt + gg + 8), (2 * cc + 9, 16 * mt + gg + 8)]
            assert [vo16[t, ch] for t, ch in order] == [base + 2 * i for i in range(8)]
    # witness: lane reads chunk L: tokens g (+8 for the second half), bands 4c..4c+3
    wo = L.w_offsets()
    for gg, cc, L_ in zip(g, c, lanes):
        for nt in range(2):
            assert [wo[8 * nt + gg, 4 * cc + i] for i in range(4)] == [L_ * 16 + 8 * nt + 2 * i for i in range(4)]
    # scales: lane (g, c) reads 4 bytes at 4g: tokens g and g + 8
    so = L.s_offsets()
    for gg in range(8):
        assert [so[gg], so[gg + 8]] == [4 * gg, 4 * gg + 2]


@pytest.mark.parametrize("m", [4, 8])
def test_key_outlier_tile_layout(m):
    """The key outlier tile is a bijection onto its fp16 slots, and lane (g, c) of the decode reads its
    tensor-core A fragment (tokens g and g + 8, columns 2c, 2c + 1 [and 2c + 8, 2c + 9]) as one word."""
    from quantized_kv_cache_kvq_gb300 import layout as L

    cols = 8 if m <= 4 else 16
    offs = L.ko_offsets(cols // 2)
    assert sorted(offs.reshape(-1).tolist()) == list(range(0, 2 * 16 * cols, 2))
    word = 8 if cols == 8 else 16
    for g in range(8):
        for c in range(4):
            lane = 4 * g + c
            base = word * lane
            assert offs[g, 2 * c] == base and offs[g, 2 * c + 1] == base + 2
            assert offs[g + 8, 2 * c] == base + 4 and offs[g + 8, 2 * c + 1] == base + 6
            if cols == 16:
                assert offs[g, 2 * c + 8] == base + 8 and offs[g + 8, 2 * c + 9] == base + 14


def test_group_scaled_int8_layouts():
    """INT8 with 32-channel scale groups: the key tile is a bijection, lane (g, c)'s 16-byte word (nt, jj) holds
    token 8nt + g in the 16-bit family's k-step order (byte 4 sidx + e <- channel 32 (2jj + (sidx >> 1)) + 8c
    + 4 (sidx & 1) + e), so the 16 channels of every k-step lie in one group; the group-scale tile is a
    bijection and lane g reads the four groups of tokens g and g + 8 as one 16-byte word."""
    from quantized_kv_cache_kvq_gb300 import layout as L

    ko = L.k_offsets("int8g32")
    assert sorted(ko.ravel().tolist()) == list(range(2048))
    for nt in range(2):
        for jj in range(2):
            for lane in range(32):
                g, c = lane >> 2, lane & 3
                word = ((nt * 2 + jj) * 32 + lane) * 16
                for sidx in range(4):
                    for e in range(4):
                        ch = 32 * (2 * jj + (sidx >> 1)) + 8 * c + 4 * (sidx & 1) + e
                        assert ko[8 * nt + g, ch] == word + 4 * sidx + e
    for jj in range(2):
        for sidx in range(4):   # k-step kb = 4jj + sidx: the channels of its 4 lanes c share one group
            chans = [32 * (2 * jj + (sidx >> 1)) + 8 * c + 4 * (sidx & 1) + e for c in range(4) for e in range(4)]
            assert len({ch // 32 for ch in chans}) == 1
            # the same channels as k-step 4jj + sidx of the 16-bit family (k-step 2j + s <- 32j + 8c + 4s + e)
            j, s = 2 * jj + (sidx >> 1), sidx & 1
            assert chans == [32 * j + 8 * c + 4 * s + e for c in range(4) for e in range(4)]
    go = L.gs_offsets()
    assert sorted((go // 2).ravel().tolist()) == list(range(64))
    for g in range(8):
        assert [go[g, k] for k in range(4)] == [16 * g + 4 * k for k in range(4)]
        assert [go[g + 8, k] for k in range(4)] == [16 * g + 4 * k + 2 for k in range(4)]


def test_group_scaled_int8_layout_combinations_refused_on_host(lib):
    import quantized_kv_cache_kvq_gb300 as kvq

    fake = 16  # aligned, never dereferenced: the layout checks come before any device work
    def cache(kf, vf, m=0):
        return kvq._Cache(k_fmt=kf, v_fmt=vf, num_kv_heads=2, num_pages=1, k_data=fake, v_data=fake, k_scale=fake,
                          v_scale=fake, witness=fake, outlier_pairs=fake if m else None, n_outlier_pairs=m,
                          k_outlier=fake if m else None)
    G32, I8, BF = kvq.FMT["int8g32"], kvq.FMT["int8"], kvq.FMT["bf16"]
    for kf, vf in ((G32, I8), (I8, G32), (BF, G32), (G32, BF)):
        c = cache(kf, vf)
        assert lib.kvq_append(ctypes.byref(c), fake, fake, 0, fake, 1, None, None) == 2, (kf, vf)
    c = cache(G32, G32, m=2)   # no outlier bypass with group scales
    assert lib.kvq_append(ctypes.byref(c), fake, fake, 0, fake, 1, None, None) == 2
    assert lib.kvq_tile_bytes(5, 0) == 0    # no format 5
