// Index arithmetic of the implicit-im2col conv factors (host and device).
//
// The patch matrix of a 3 x 3, stride 1, zero padding 1 convolution over NHWC
// activations has one row per output position (n, h, w), in that order, and
// columns (dh*3 + dw)*C + c followed by one ones column (the bias).  The
// factor kernel reads it in 64-column boxes and 64-row k-blocks:
//   * box q (columns 64q .. 64q + 63) is, for C % 64 == 0, channels
//     c0 .. c0 + 63 of tap (dh, dw) when q < 9C/64, the bias column when
//     q == 9C/64, and past d otherwise (conv_box_source);
//   * the k-blocks of a worker start at positions 0, 64, 128, ..., stepped
//     without division by carrying 64 = sn*H*W + sh*W + sw (conv_step).
#pragma once

namespace kfac {

struct ConvGeom {
  int c64, H, W;   // channels / 64, image height and width
  int sw, sh, sn;  // `rows` positions = sn images + sh rows + sw columns
};

__host__ __device__ inline ConvGeom make_conv_geom(int C, int H, int W, int rows) {
  const int along_w = rows / W;
  return ConvGeom{C / 64, H, W, rows % W, along_w % H, along_w / H};
}

// (n, h, w) -> the position `rows` further on (rows as given to make_conv_geom).
__host__ __device__ inline void conv_step(const ConvGeom& g, int& n, int& h, int& w) {
  w += g.sw;
  if (w >= g.W) {
    w -= g.W;
    ++h;
  }
  h += g.sh;
  if (h >= g.H) {
    h -= g.H;
    ++n;
  }
  n += g.sn;
}

struct ConvBox {
  int c0, dw, dh;
  int kind;  // 0 tap (channels c0.., offsets dh, dw), 1 bias column, 2 past d
};

__host__ __device__ inline ConvBox conv_box_source(const ConvGeom& g, int q) {
  ConvBox b{0, 0, 0, q == 9 * g.c64 ? 1 : 2};
  if (q < 9 * g.c64) {
    const int tap = q / g.c64;
    b.dh = tap / 3;
    b.dw = tap - 3 * b.dh;
    b.c0 = (q - tap * g.c64) * 64;
    b.kind = 0;
  }
  return b;
}

}  // namespace kfac
