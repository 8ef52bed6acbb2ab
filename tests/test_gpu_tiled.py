"""Tiled decode (vae_decode_chain_tiled) against the float64 oracle's tiled
decode (cortiq-engine 0.8.78, vae3d.rs: split_tiles / blend / crop /
decode_clip, applied to this decoder): the same tile schedule, each tile's
latent crop decoded on its own, the tiles cross-faded over their overlaps.
The bar is the decoder's RGB bar (cosine >= 0.99999, max |err| <= 5e-3)."""
import numpy as np
import pytest

import oracle as O
import vae_synth as S
from tests._parity import COS_MIN, RGB_MAXABS, SENTINEL, assert_all_written, metrics

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import diffusion_vae_decoder_gb300 as p
    p.load_library()
    yield p
    assert p.vae_device_error() == 0


def _tiled(pkg, arch, latent, seed, tile, overlap, batch):
    w = S.make_decoder_weights(arch, seed)
    z = S.make_latent(latent, seed)
    chain = pkg.VaeChain(w, n_up_blocks=4)
    n, _, h, ww = latent
    out = torch.full((n, 3, 8 * h, 8 * ww), SENTINEL, device="cuda")
    chain.decode_tiled(torch.from_numpy(z).cuda(), tile=tile, min_overlap=overlap,
                       tiles_per_batch=batch, out=out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    chain.close()
    return w, z, got


def _check(got, ref, what):
    assert_all_written(got, what)
    m = metrics(got, ref)
    print(what, m)
    assert m["cos"] >= COS_MIN and m["max_abs"] <= RGB_MAXABS, (what, m)


def test_tiled_tiny_decoder_two_images_ragged_batches(pkg):
    """96 x 160 output in 64-pixel tiles (2 x 3 per image, overlaps 32 and
    16), two images, decoded five tiles at a time (batches cross images)."""
    w, z, got = _tiled(pkg, "tiny", (2, 16, 12, 20), 81, 64, 16, 5)
    ref = O.tiled_decode(z, w, S.SCALING_FACTOR, S.SHIFT_FACTOR, 4, tile=64, min_overlap=16)
    _check(got, ref, "tiled tiny [2,16,12,20]")


def test_tiled_flux_decoder(pkg):
    """320 x 288 output in 256-pixel tiles (2 x 2, overlaps 192 and 224)."""
    w, z, got = _tiled(pkg, "flux", (1, 16, 40, 36), 82, 256, 64, 2)
    ref = O.tiled_decode(z, w, S.SCALING_FACTOR, S.SHIFT_FACTOR, 4, tile=256, min_overlap=64)
    _check(got, ref, "tiled flux [1,16,40,36]")


def test_one_tile_is_the_whole_decode_bit_for_bit(pkg):
    w = S.make_decoder_weights("flux", 83)
    z = torch.from_numpy(S.make_latent((1, 16, 16, 24), 83)).cuda()
    chain = pkg.VaeChain(w, n_up_blocks=4)
    a = chain.decode(z)
    b = chain.decode_tiled(z, tile=256, min_overlap=64, tiles_per_batch=1)
    torch.cuda.synchronize()
    chain.close()
    assert torch.equal(a, b)


def test_output_beyond_the_whole_image_limit(pkg):
    """A 272 x 272 latent (73984 tokens, above the 65536 the whole-image
    decode accepts) decodes as 5 x 5 tiles of 512 pixels, four per batch.
    Every pixel is written; the kept part of the first tile (no neighbour
    above or to the left) is that tile's decode, checked against the
    oracle."""
    seed = 84
    w = S.make_decoder_weights("flux", seed)
    zn = S.make_latent((1, 16, 272, 272), seed)
    z = torch.from_numpy(zn).cuda()
    chain = pkg.VaeChain(w, n_up_blocks=4)
    rgb = torch.empty((1, 3, 2176, 2176), device="cuda")
    ws = torch.empty(chain.workspace_size(1, 128, 128), dtype=torch.uint8, device="cuda")
    with pytest.raises(pkg.VaeError) as e:
        chain.decode(z, out=rgb, ws=ws)
    assert e.value.status == -2
    del ws
    rgb.fill_(SENTINEL)
    chain.decode_tiled(z, tile=512, min_overlap=64, tiles_per_batch=4, out=rgb)
    torch.cuda.synchronize()
    chain.close()
    got = rgb.cpu().numpy()
    assert_all_written(got, "tiled 2176^2")
    assert np.isfinite(got).all()
    ys, _, yo = O.split_tiles(2176, 8, 512, 64)
    assert len(ys) == 5
    keep = 512 - yo[0]
    ref = O.decode(zn[:, :, :64, :64], w, S.SCALING_FACTOR, S.SHIFT_FACTOR, 4)
    _check(got[:, :, :keep, :keep], ref[:, :, :keep, :keep], "tiled 2176^2, first tile")
