"""Host-side checks of the Mimi decoder's binding (no GPU): the canonical tensor order of
include/pm_mimi.h as the binding states it, as the seeded generator draws it and as the
oracle reads it are the same list; the config struct mirrors the C layout; the library
counts the tensors and refuses configurations its kernels do not take."""
import ctypes as C

from full_duplex_speech_moshi_gb300 import inputs as I
from full_duplex_speech_moshi_gb300 import pm
from oracle import mimi as M


def test_three_statements_of_the_tensor_order_agree():
    for shape in (I.MIMI_SMALL, I.MIMI_FULL):
        gen = I.mimi_tensor_specs(shape)
        orc = [(n, tuple(s)) for n, s in M.tensor_specs(M.MimiShape(**shape))]
        assert gen == orc
        assert [n for n, _ in gen] == pm.mimi_tensor_names(shape)
        cfg = pm.make_mimi_config(shape, B_max=1)
        assert pm.lib().pm_mimi_tensor_count(C.byref(cfg)) == len(gen)


def test_full_shape_frame():
    assert pm.mimi_frame_samples(I.MIMI_FULL) == 1920  # 80 ms at 24 kHz
    assert len(I.mimi_tensor_specs(I.MIMI_FULL)) == 8 + 3 + 80 + 2 + 24 + 2


def test_config_struct_layout():
    assert C.sizeof(pm.pm_mimi_config) == 4 * (11 + pm.PM_MIMI_MAX_RATIOS + 6 + 2)


def test_unsupported_configurations_are_refused():
    L = pm.lib()
    for over in (dict(dim=320, heads=5), dict(dim=512, heads=4), dict(up_kernel=6), dict(up_stride=3),
                 dict(n_q=1), dict(n_q=17), dict(cb_dim=12), dict(ratios=[]), dict(ratios=[8, 0]),
                 dict(ffn=1000), dict(ln_eps=0.0), dict(compress=3)):
        cfg = pm.make_mimi_config(dict(I.MIMI_FULL, **over), B_max=1)
        assert L.pm_mimi_tensor_count(C.byref(cfg)) == -1, over
    for B in (0, 9):
        assert L.pm_mimi_tensor_count(C.byref(pm.make_mimi_config(I.MIMI_FULL, B_max=B))) == -1


def test_generator_draws_are_seeded_and_scaled():
    a = I.make_mimi_weights(I.MIMI_SMALL)
    b = I.make_mimi_weights(I.MIMI_SMALL)
    assert all((a[k] == b[k]).all() for k in a)
    w = I.bf16_bits_to_f32(I.make_mimi_weights(I.MIMI_FULL)["dec.up0.w"])  # [1024][512][16]: fan 512 x 16
    assert abs(w.std() * (512 * 16) ** 0.5 - 1.0) < 0.01
    c = I.make_mimi_codes(I.MIMI_FULL, 50, 2)
    assert c.shape == (50, 2, 8) and c.min() >= 0 and c.max() < 2048


def test_encoder_tensor_order_agrees():
    for shape in (I.MIMI_SMALL, I.MIMI_FULL):
        gen = I.mimi_encoder_tensor_specs(shape)
        orc = [(n, tuple(s)) for n, s in M.encoder_tensor_specs(M.MimiShape(**shape))]
        assert gen == orc
        assert [n for n, _ in gen] == pm.mimi_encoder_tensor_names(shape)
        cfg = pm.make_mimi_config(shape, B_max=1)
        assert pm.lib().pm_mimi_encoder_tensor_count(C.byref(cfg)) == len(gen)
    # the encoder's own limits: codebooks split over 8 CTAs
    cfg = pm.make_mimi_config(dict(I.MIMI_SMALL, card=60), B_max=1)
    assert pm.lib().pm_mimi_encoder_tensor_count(C.byref(cfg)) == -1
    assert pm.lib().pm_mimi_tensor_count(C.byref(cfg)) > 0
