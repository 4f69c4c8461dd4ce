// Host side of the C ABI: offline packers, blob validation, handles.
//
// The packers turn canonical arrays into the device layouts described in
// q2_layout.h.  They run once per matrix, off the timed path (the pages'
// load-time repack: "Qwen3-8B -- 2-bit BPDQ (packed)", Format: at load the
// packed tensors are repacked, not decoded; "Unfolding the Leech Lattice",
// section 2: offline expansion into divergence-free GPU layouts).
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "q2_internal.h"

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Builder {
  q2_blob_header hdr;
  size_t cursor;
  Builder(int fmt, int R, int C) {
    std::memset(&hdr, 0, sizeof(hdr));
    hdr.magic = Q2_MAGIC;
    hdr.version = Q2_VERSION;
    hdr.fmt = fmt;
    hdr.R = R;
    hdr.C = C;
    hdr.Rpad = (R + Q2_ROWS - 1) / Q2_ROWS * Q2_ROWS;
    cursor = align_up(sizeof(q2_blob_header), kAlign);
  }
  void section(int i, size_t bytes) {
    hdr.off[i] = cursor;
    hdr.len[i] = bytes;
    cursor = align_up(cursor + bytes, kAlign);
  }
  size_t total() {
    hdr.total_bytes = cursor;
    return cursor;
  }
};

// Two-phase protocol: size query or fill.  Returns Q2_OK and sets *out_bytes.
int finish(Builder& b, void* out, size_t* out_bytes, bool* fill) {
  size_t tot = b.total();
  if (!out) {
    *out_bytes = tot;
    *fill = false;
    return Q2_OK;
  }
  if (*out_bytes < tot) {
    *out_bytes = tot;
    return Q2_ESIZE;
  }
  std::memset(out, 0, tot);
  std::memcpy(out, &b.hdr, sizeof(b.hdr));
  *out_bytes = tot;
  *fill = true;
  return Q2_OK;
}

unsigned char* sec(void* out, const q2_blob_header& h, int i) {
  return static_cast<unsigned char*>(out) + h.off[i];
}

// Exact fp16 <-> double conversions (host; IEEE binary16).
double half_to_double(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 0) v = std::ldexp((double)m, -24);
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = std::ldexp((double)(m | 1024), e - 25);
  return s ? -v : v;
}

uint16_t double_to_half_rne(double d) {
  // Round-to-nearest-even of a finite double to binary16.
  uint16_t sign = std::signbit(d) ? 0x8000 : 0;
  double a = std::fabs(d);
  if (std::isnan(d)) return 0x7e00;
  if (a >= 65520.0) return sign | 0x7c00;
  if (a < std::ldexp(1.0, -25)) {
    // below half the smallest subnormal; exactly half rounds to even (0)
    return sign;
  }
  int e;
  std::frexp(a, &e);       // a = f * 2^e, f in [0.5, 1)
  int exp = e - 1;         // a = 1.x * 2^exp
  if (exp < -14) exp = -14;  // subnormal range uses fixed exponent
  // quantum = 2^(exp - 10)
  double q = std::ldexp(1.0, exp - 10);
  double n = a / q;        // exact (power-of-two scaling)
  double r = std::nearbyint(n);   // default rounding mode: nearest-even
  uint32_t mant = (uint32_t)r;
  if (mant >= 2048) {      // carried into the next binade
    mant >>= 1;
    exp += 1;
  }
  if (exp > 15) return sign | 0x7c00;
  if (mant < 1024) return sign | (uint16_t)mant;            // subnormal
  return sign | (uint16_t)(((exp + 15) << 10) | (mant - 1024));
}

}  // namespace

extern "C" {

const char* q2_strerror(int status) {
  switch (status) {
    case Q2_OK: return "ok";
    case Q2_EINVAL: return "invalid argument";
    case Q2_ESHAPE: return "shape not accepted by this format";
    case Q2_EALIGN: return "pointer not 16-byte aligned";
    case Q2_EFMT: return "format does not match the handle";
    case Q2_ENTOK: return "ntok outside 1..64";
    case Q2_EBLOB: return "blob header corrupt or wrong version";
    case Q2_EWORKSPACE: return "workspace missing or too small";
    case Q2_ECUDA: return "CUDA call or kernel launch failed";
    case Q2_ENOMEM: return "host allocation failed";
    case Q2_ESIZE: return "output buffer too small";
    case Q2_ESCRATCH: return "problem larger than the built-in scratch (Q2_NOALLOC_SCRATCH_BYTES)";
    default: return "unknown status";
  }
}

int q2_pack_fp16(const uint16_t* w, int R, int C, void* out, size_t* out_bytes) {
  if (!out_bytes || (out && !w)) return Q2_EINVAL;
  if (R < 1 || C < 8 || C % 8) return Q2_ESHAPE;
  Builder b(Q2_FP16, R, C);
  b.section(SEC_FP16_W, (size_t)R * C * 2);
  bool fill;
  int st = finish(b, out, out_bytes, &fill);
  if (st || !fill) return st;
  std::memcpy(sec(out, b.hdr, SEC_FP16_W), w, (size_t)R * C * 2);
  return Q2_OK;
}

int q2_pack_bpdq(const uint8_t* plane0, const uint8_t* plane1, const uint16_t* coef,
                 int R, int C, void* out, size_t* out_bytes) {
  if (!out_bytes || (out && (!plane0 || !plane1 || !coef))) return Q2_EINVAL;
  if (R < 1 || C < Q2_SLICE || C % Q2_SLICE) return Q2_ESHAPE;
  Builder b(Q2_BPDQ, R, C);
  const int G = C / Q2_SLICE, Rp = b.hdr.Rpad, nrb = Rp / Q2_ROWS;
  b.hdr.nslice = G;
  b.section(SEC_BPDQ_BITS, (size_t)G * nrb * Q2_ITEM_BYTES_BPDQ);
  b.section(SEC_BPDQ_C01, (size_t)G * Rp * 4);
  b.section(SEC_BPDQ_OFF, (size_t)G * Rp * 2);
  b.section(SEC_BPDQ_VTAB, (size_t)G * Rp * 8);
  bool fill;
  int st = finish(b, out, out_bytes, &fill);
  if (st || !fill) return st;
  const size_t rowbytes = (size_t)C / 8;
  unsigned char* bits = sec(out, b.hdr, SEC_BPDQ_BITS);
  for (int g = 0; g < G; ++g)
    for (int rb = 0; rb < nrb; ++rb) {
      unsigned char* item = bits + ((size_t)g * nrb + rb) * Q2_ITEM_BYTES_BPDQ;
      for (int k = 0; k < 4; ++k) {
        const uint8_t* plane = (k < 2) ? plane0 : plane1;
        for (int l = 0; l < 32; ++l) {
          const int r = rb * 32 + l;
          if (r >= R) continue;
          for (int q = 0; q < 16; ++q) {
            const int P = (k & 1) * 16 + q;
            const int beta = (P + l) & 31;
            item[k * 512 + l * 16 + q] = plane[(size_t)r * rowbytes + (size_t)g * 32 + beta];
          }
        }
      }
    }
  uint16_t* c01 = reinterpret_cast<uint16_t*>(sec(out, b.hdr, SEC_BPDQ_C01));
  uint16_t* offs = reinterpret_cast<uint16_t*>(sec(out, b.hdr, SEC_BPDQ_OFF));
  uint16_t* vtab = reinterpret_cast<uint16_t*>(sec(out, b.hdr, SEC_BPDQ_VTAB));
  for (int g = 0; g < G; ++g)
    for (int r = 0; r < R; ++r) {
      const uint16_t* cf = coef + ((size_t)g * R + r) * 3;
      const size_t i = (size_t)g * Rp + r;
      c01[2 * i] = cf[0];
      c01[2 * i + 1] = cf[1];
      offs[i] = cf[2];
      // value table: code k = b0 | b1 << 1 -> one rounding of the exact sum
      const double c0 = half_to_double(cf[0]), c1 = half_to_double(cf[1]), of = half_to_double(cf[2]);
      for (int k = 0; k < 4; ++k)
        vtab[4 * i + k] = double_to_half_rne(of + ((k & 1) ? c0 : 0.0) + ((k & 2) ? c1 : 0.0));
    }
  return Q2_OK;
}

int q2_pack_trellis(const uint8_t* stream, const uint16_t* table, const uint16_t* scale,
                    int R, int C, void* out, size_t* out_bytes) {
  if (!out_bytes || (out && (!stream || !table || !scale))) return Q2_EINVAL;
  if (R < 1 || C < Q2_SLICE || C % Q2_SLICE) return Q2_ESHAPE;
  Builder b(Q2_TRELLIS, R, C);
  const int S = C / Q2_SLICE, Rp = b.hdr.Rpad, nrb = Rp / Q2_ROWS;
  b.hdr.nslice = S;
  b.section(SEC_TRL_STREAM, (size_t)S * nrb * Q2_ITEM_BYTES_TRL);
  b.section(SEC_TRL_TABLE, 4096 * 2 * 2);
  b.section(SEC_TRL_SCALE, (size_t)Rp * 2);
  bool fill;
  int st = finish(b, out, out_bytes, &fill);
  if (st || !fill) return st;
  unsigned char* dst = sec(out, b.hdr, SEC_TRL_STREAM);
  for (int s = 0; s < S; ++s)
    for (int rb = 0; rb < nrb; ++rb) {
      unsigned char* item = dst + ((size_t)s * nrb + rb) * Q2_ITEM_BYTES_TRL;
      for (int l = 0; l < 32; ++l) {
        const int r = rb * 32 + l;
        if (r >= R) continue;
        const uint8_t* seg = stream + ((size_t)r * S + s) * 64;
        unsigned char lane[64];
        std::memset(lane, 0, 64);
        for (int n = 0; n < 128; ++n) {
          const int k = 127 - n;   // nibble n holds symbol 127 - n
          const int sym = (k & 1) ? (seg[k >> 1] >> 4) : (seg[k >> 1] & 15);
          lane[n >> 1] |= (unsigned char)(sym << ((n & 1) * 4));
        }
        for (int w = 0; w < 16; ++w) {
          const int k = w >> 2;   // chunk
          std::memcpy(item + k * 512 + l * 16 + (w & 3) * 4, lane + w * 4, 4);
        }
      }
    }
  std::memcpy(sec(out, b.hdr, SEC_TRL_TABLE), table, 4096 * 2 * 2);
  std::memcpy(sec(out, b.hdr, SEC_TRL_SCALE), scale, (size_t)R * 2);
  return Q2_OK;
}

int q2_pack_leech(const int8_t* v, const uint16_t* tail, const uint16_t* scale,
                  int R, int C, float inv_sqrt8, int layout, void* out, size_t* out_bytes) {
  if (!out_bytes || (out && (!v || !scale || (C % 24 && !tail)))) return Q2_EINVAL;
  if (layout != Q2_LEECH_PLANES3 && layout != Q2_LEECH_OFFSET4) return Q2_EINVAL;
  if (R < 1 || C < 24) return Q2_ESHAPE;
  const bool off4 = layout == Q2_LEECH_OFFSET4;
  const int NP = off4 ? 4 : 3;
  const int item_bytes = off4 ? Q2_ITEM_BYTES_LEECH4 : Q2_ITEM_BYTES_LEECH;
  Builder b(Q2_LEECH, R, C);
  b.hdr.layout = layout;
  const int nb = C / 24, TL = C % 24, TLp = (TL + 7) / 8 * 8;
  const int S = (C + Q2_SLICE - 1) / Q2_SLICE, Rp = b.hdr.Rpad, nrb = Rp / Q2_ROWS;
  b.hdr.nslice = S;
  b.hdr.nblock = nb;
  b.hdr.tail = TL;
  b.hdr.tailpad = TLp;
  b.hdr.inv_sqrt8 = inv_sqrt8;
  // validate and count exceptions first
  uint32_t nexc = 0;
  if (out) {
    for (size_t i = 0; i < (size_t)R * nb; ++i) {
      const int8_t* blk = v + i * 24;
      const int p = blk[0] & 1;
      for (int j = 0; j < 24; ++j) {
        if ((blk[j] & 1) != p || blk[j] < -8 || blk[j] > 8) return Q2_EINVAL;
        if (blk[j] == 8 && !off4) ++nexc;
      }
    }
  }
  b.section(SEC_LEECH_PLANES, (size_t)S * nrb * item_bytes);
  b.section(SEC_LEECH_PARITY, (size_t)S * Rp * 2);
  b.section(SEC_LEECH_SCALE, (size_t)Rp * 2);
  b.section(SEC_LEECH_TAIL, (size_t)Rp * TLp * 2);
  b.section(SEC_LEECH_EXCPTR, (size_t)(Rp + 1) * 4);
  if (!out) {
    // size query: reserve the worst case for the exception list is not
    // possible without the data; callers pass v on the query as well.
    uint32_t q = 0;
    if (v && !off4) {
      for (size_t i = 0; i < (size_t)R * nb * 24; ++i) q += (v[i] == 8);
    }
    nexc = q;
  }
  b.hdr.nexc = nexc;
  b.section(SEC_LEECH_EXCCOL, (size_t)nexc * 4);
  bool fill;
  int st = finish(b, out, out_bytes, &fill);
  if (st || !fill) return st;
  // canonical per-row planes (bit c of a [C/8 padded to S*32] byte row)
  const size_t rowbytes = (size_t)S * 32;
  std::vector<uint8_t> pl[4];
  for (int p = 0; p < NP; ++p) pl[p].assign(rowbytes, 0);
  unsigned char* planes = sec(out, b.hdr, SEC_LEECH_PLANES);
  uint16_t* parity = reinterpret_cast<uint16_t*>(sec(out, b.hdr, SEC_LEECH_PARITY));
  uint32_t* excptr = reinterpret_cast<uint32_t*>(sec(out, b.hdr, SEC_LEECH_EXCPTR));
  uint32_t* exccol = reinterpret_cast<uint32_t*>(sec(out, b.hdr, SEC_LEECH_EXCCOL));
  uint32_t ne = 0;
  for (int r = 0; r < Rp; ++r) {
    excptr[r] = ne;
    if (r >= R && !off4) continue;
    for (int p = 0; p < NP; ++p) std::fill(pl[p].begin(), pl[p].end(), 0);
    // offset binary: every column outside the blocks (tail, padding columns,
    // padding rows) holds code 4, the code of 0, so the -8 offset cancels there
    if (off4) std::fill(pl[2].begin(), pl[2].end(), (uint8_t)0xFF);
    const int nbr = r < R ? nb : 0;             // padding rows: no blocks
    std::vector<uint16_t> par(S, 0);
    for (int bk = 0; bk < nbr; ++bk) {
      const int8_t* blk = v + ((size_t)r * nb + bk) * 24;
      const int p = blk[0] & 1;
      const int c0 = bk * 24;
      const int sl = c0 / Q2_SLICE;
      const int first = (sl * Q2_SLICE + 23) / 24;   // first block starting in slice sl
      if (p) par[sl] |= (uint16_t)(1u << (bk - first));
      for (int j = 0; j < 24; ++j) {
        int val = blk[j];
        int code;
        if (off4) {
          code = (val - p) / 2 + 4;         // offset binary, 0..8
        } else {
          if (val == 8) {
            exccol[ne++] = (uint32_t)(c0 + j);
            val = -8;
          }
          code = ((val - p) / 2) & 7;       // u in [-4, 3], three-bit two's complement
        }
        const int c = c0 + j;
        for (int q = 0; q < NP; ++q) {
          const uint8_t bit = (uint8_t)(1u << (c & 7));
          pl[q][c >> 3] = ((code >> q) & 1) ? (uint8_t)(pl[q][c >> 3] | bit) : (uint8_t)(pl[q][c >> 3] & ~bit);
        }
      }
    }
    for (int s = 0; s < S; ++s) parity[(size_t)s * Rp + r] = r < R ? par[s] : (uint16_t)0;
    const int rb = r / 32, l = r % 32;
    for (int s = 0; s < S; ++s) {
      unsigned char* item = planes + ((size_t)s * nrb + rb) * item_bytes;
      for (int k = 0; k < 2 * NP; ++k)
        for (int q = 0; q < 16; ++q) {
          const int P = (k & 1) * 16 + q;
          const int beta = (P + l) & 31;
          item[k * 512 + l * 16 + q] = pl[k >> 1][(size_t)s * 32 + beta];
        }
    }
  }
  excptr[Rp] = ne;
  uint16_t* sc = reinterpret_cast<uint16_t*>(sec(out, b.hdr, SEC_LEECH_SCALE));
  std::memcpy(sc, scale, (size_t)R * 2);
  uint16_t* tl = reinterpret_cast<uint16_t*>(sec(out, b.hdr, SEC_LEECH_TAIL));
  for (int r = 0; r < R; ++r)
    for (int j = 0; j < TL; ++j) tl[(size_t)r * TLp + j] = tail[(size_t)r * TL + j];
  return Q2_OK;
}

int q2_pack_noweights(int R, int C, void* out, size_t* out_bytes) {
  if (!out_bytes) return Q2_EINVAL;
  if (R < 1 || C < Q2_SLICE || C % Q2_SLICE) return Q2_ESHAPE;
  Builder b(Q2_NOWEIGHTS, R, C);
  b.hdr.nslice = C / Q2_SLICE;
  bool fill;
  return finish(b, out, out_bytes, &fill);
}

// Bound on |one slice's partial sum| over any fp16 x (|x| <= 65504), from
// the largest per-weight magnitude of the matrix: 256 columns x 65504 x
// max |w| (before the row scale, which the epilogue applies).
static double partial_bound(const unsigned char* blob, const q2_blob_header& d) {
  double k = 0.0;
  switch (d.fmt) {
    case Q2_BPDQ: {
      const uint16_t* c01 = reinterpret_cast<const uint16_t*>(blob + d.off[SEC_BPDQ_C01]);
      const uint16_t* off = reinterpret_cast<const uint16_t*>(blob + d.off[SEC_BPDQ_OFF]);
      const size_t n = (size_t)d.nslice * d.Rpad;
      for (size_t i = 0; i < n; ++i) {
        const double v = std::fabs(half_to_double(c01[2 * i])) + std::fabs(half_to_double(c01[2 * i + 1])) +
                         std::fabs(half_to_double(off[i]));
        if (v > k) k = v;
      }
      break;
    }
    case Q2_TRELLIS: {
      const uint16_t* t = reinterpret_cast<const uint16_t*>(blob + d.off[SEC_TRL_TABLE]);
      for (int i = 0; i < 4096 * 2; ++i) k = std::fmax(k, std::fabs(half_to_double(t[i])));
      break;
    }
    case Q2_LEECH: k = 8.0; break;          // |v| <= 8 per coordinate
    case Q2_NOWEIGHTS: k = 0.04; break;     // the control's synthetic coefficients
    default: k = 0.0;
  }
  if (!(k < 1e30)) k = 1e30;                // inf / nan coefficients: keep the scale finite
  return k * 256.0 * 65504.0;
}

int q2_bind(const void* blob_host, const void* blob_dev, q2_handle** h) {
  if (!blob_host || !blob_dev || !h) return Q2_EINVAL;
  if (reinterpret_cast<uintptr_t>(blob_dev) % kAlign) return Q2_EALIGN;
  q2_blob_header hdr;
  std::memcpy(&hdr, blob_host, sizeof(hdr));
  if (hdr.magic != Q2_MAGIC || hdr.version != Q2_VERSION) return Q2_EBLOB;
  if (hdr.fmt < Q2_FP16 || hdr.fmt > Q2_NOWEIGHTS || hdr.R < 1 || hdr.C < 1 ||
      hdr.Rpad != (hdr.R + 31) / 32 * 32)
    return Q2_EBLOB;
  for (int i = 0; i < Q2_MAX_SECTIONS; ++i)
    if (hdr.len[i] && (hdr.off[i] % kAlign || hdr.off[i] + hdr.len[i] > hdr.total_bytes)) return Q2_EBLOB;
  if (hdr.layout != 0 && !(hdr.fmt == Q2_LEECH && hdr.layout == Q2_LEECH_OFFSET4)) return Q2_EBLOB;
  q2_handle* p = new (std::nothrow) q2_handle;
  if (!p) return Q2_ENOMEM;
  p->hdr = hdr;
  p->dev = static_cast<const unsigned char*>(blob_dev);
  p->ws = nullptr;
  p->ws_bytes = 0;
  p->pbound = partial_bound(static_cast<const unsigned char*>(blob_host), hdr);
  *h = p;
  return Q2_OK;
}

void q2_unbind(q2_handle* h) { delete h; }

extern "C" size_t q2_tc_workspace_bytes(const q2_handle* h, int ntok);   // q2_tc.cu

int q2_workspace_bytes(const q2_handle* h, int ntok, size_t* bytes) {
  if (!h || !bytes) return Q2_EINVAL;
  if (ntok < 1 || ntok > Q2_MAX_NTOK) return Q2_ENTOK;
  const int fmt = h->hdr.fmt;
  if (fmt == Q2_FP16) {                                        // one token: none; more: the tensor-core plan
    *bytes = ntok == 1 ? 0 : q2_tc_workspace_bytes(h, ntok);
    return Q2_OK;
  }
  const bool cuda_core = ntok == 1 || (fmt == Q2_BPDQ && ntok <= Q2_MAX_ACC_TOK) ||
                         (fmt == Q2_LEECH && ntok == 2 && h->hdr.C % 8 == 0 && h->hdr.R % 8 == 0);
  if (cuda_core)
    *bytes = (size_t)ntok * h->hdr.Rpad * 8;                 // accumulators
  else
    *bytes = q2_tc_workspace_bytes(h, ntok);                  // the tensor-core launch's plan
  return Q2_OK;
}

int q2_set_workspace(q2_handle* h, void* ws_dev, size_t ws_bytes) {
  if (!h) return Q2_EINVAL;
  if (ws_dev && reinterpret_cast<uintptr_t>(ws_dev) % kAlign) return Q2_EALIGN;
  h->ws = ws_dev;
  h->ws_bytes = ws_dev ? ws_bytes : 0;
  return Q2_OK;
}

int q2_info(const q2_handle* h, int* fmt, int* R, int* C) {
  if (!h) return Q2_EINVAL;
  if (fmt) *fmt = h->hdr.fmt;
  if (R) *R = h->hdr.R;
  if (C) *C = h->hdr.C;
  return Q2_OK;
}

int q2_bytes(const q2_handle* h, int ntok, size_t* bytes) {
  if (!h || !bytes) return Q2_EINVAL;
  if (ntok < 1 || ntok > Q2_MAX_NTOK) return Q2_ENTOK;
  const q2_blob_header& d = h->hdr;
  switch (d.fmt) {
    case Q2_FP16: *bytes = d.len[SEC_FP16_W]; break;
    case Q2_BPDQ:
      // batch 1 reads (c0, c1, off); the multi-token path reads the value table
      *bytes = d.len[SEC_BPDQ_BITS] + (ntok == 1 ? d.len[SEC_BPDQ_C01] + d.len[SEC_BPDQ_OFF]
                                                 : d.len[SEC_BPDQ_VTAB]);
      break;
    case Q2_TRELLIS:
      *bytes = d.len[SEC_TRL_STREAM] + d.len[SEC_TRL_TABLE] + d.len[SEC_TRL_SCALE];
      break;
    case Q2_LEECH:
      *bytes = d.len[SEC_LEECH_PLANES] + d.len[SEC_LEECH_PARITY] + d.len[SEC_LEECH_SCALE] +
               d.len[SEC_LEECH_TAIL] + d.len[SEC_LEECH_EXCPTR] + d.len[SEC_LEECH_EXCCOL];
      break;
    default: *bytes = 0;
  }
  return Q2_OK;
}

int q2_decode_bytes(const q2_handle* h, size_t* bytes) {
  if (!h || !bytes) return Q2_EINVAL;
  const q2_blob_header& d = h->hdr;
  switch (d.fmt) {
    case Q2_FP16:
    case Q2_BPDQ: *bytes = (size_t)d.R * d.C * 2; break;
    case Q2_TRELLIS: *bytes = (size_t)d.R * d.C * 4; break;
    case Q2_LEECH: {
      size_t body = (size_t)d.R * d.nblock * 24;
      body = (body + 15) / 16 * 16;
      *bytes = body + (size_t)d.R * d.tail * 2;
      break;
    }
    default: return Q2_EFMT;
  }
  return Q2_OK;
}

static int gemv_impl(q2_fmt fmt, const q2_handle* h, const void* x, void* y, int ntok, q2_stream stream,
                     const q2_pf* pf) {
  if (!h || !x || !y) return Q2_EINVAL;
  if ((int)fmt != h->hdr.fmt) return Q2_EFMT;
  if (ntok < 1 || ntok > Q2_MAX_NTOK) return Q2_ENTOK;
  if (reinterpret_cast<uintptr_t>(x) % 16 || reinterpret_cast<uintptr_t>(y) % 16) return Q2_EALIGN;
  size_t need = 0;
  int st = q2_workspace_bytes(h, ntok, &need);
  if (st) return st;
  if (need && (!h->ws || h->ws_bytes < need)) return Q2_EWORKSPACE;
  if (h->hdr.Rpad > Q2_MAX_ROWS || h->hdr.nslice > Q2_MAX_SPLIT) return Q2_ESHAPE;
  void* s = static_cast<void*>(stream);
  switch (h->hdr.fmt) {
    case Q2_FP16: return q2_launch_fp16(h, x, y, ntok, s, pf);
    case Q2_BPDQ: return q2_launch_bpdq(h, x, y, ntok, s, pf);
    case Q2_TRELLIS: return q2_launch_trellis(h, x, y, ntok, s, pf);
    case Q2_LEECH: return q2_launch_leech(h, x, y, ntok, s, pf);
    case Q2_NOWEIGHTS: return q2_launch_noweights(h, x, y, ntok, s, pf);
    default: return Q2_EFMT;
  }
}

int q2_gemv(q2_fmt fmt, const q2_handle* h, const void* x, void* y, int ntok, q2_stream stream) {
  return gemv_impl(fmt, h, x, y, ntok, stream, nullptr);
}

// The device bytes a GEMV of h reads at ntok tokens on the CUDA-core path,
// as one range from its first weight section to the end of the last one it
// reads (the holes between sections are alignment padding, under 256 bytes
// each).  Zero length for the no-weights control.
static void weight_range(const q2_handle* h, int ntok, const unsigned char** p, unsigned long long* n) {
  const q2_blob_header& d = h->hdr;
  int last = -1;
  switch (d.fmt) {
    case Q2_FP16: last = SEC_FP16_W; break;
    case Q2_BPDQ: last = ntok <= Q2_MAX_ACC_TOK ? SEC_BPDQ_OFF : -1; break;
    case Q2_TRELLIS: last = ntok == 1 ? SEC_TRL_SCALE : -1; break;
    case Q2_LEECH: last = ntok == 1 ? SEC_LEECH_EXCCOL : -1; break;
    default: last = -1;
  }
  *p = h->dev + d.off[0];
  *n = 0;
  for (int s = last; s >= 0; --s)
    if (d.len[s]) {                       // the last non-empty section ends the range
      *n = (d.off[s] + d.len[s] - d.off[0]) / 16 * 16;
      break;
    }
}

int q2_gemv_chain(int n, const q2_fmt* fmt, q2_handle* const* h, const void* const* x, void* const* y, int ntok,
                  int lookahead, q2_stream stream) {
  if (n < 0 || (n > 0 && (!fmt || !h || !x || !y))) return Q2_EINVAL;
  if (lookahead < 0 || lookahead > Q2_PF_SLOTS) return Q2_EINVAL;
  for (int i = 0; i < n; ++i) {               // refuse the whole chain before launching any of it
    if (!h[i] || !x[i] || !y[i]) return Q2_EINVAL;
    if ((int)fmt[i] != h[i]->hdr.fmt) return Q2_EFMT;
  }
  for (int i = 0; i < n; ++i) {
    // launch 0 fetches GEMVs 1..lookahead, launch i > 0 only GEMV i + lookahead
    // (the ones in between were fetched by the launches before it)
    q2_pf pf = {};
    for (int k = (i == 0 ? 1 : lookahead), slot = 0; k <= lookahead && i + k < n; ++k, ++slot)
      weight_range(h[i + k], ntok, &pf.ptr[slot], &pf.len[slot]);
    const int st = gemv_impl(fmt[i], h[i], x[i], y[i], ntok, stream, lookahead ? &pf : nullptr);
    if (st) return st;
  }
  return Q2_OK;
}

int q2_decode(const q2_handle* h, void* out_dev, q2_stream stream) {
  if (!h || !out_dev) return Q2_EINVAL;
  if (h->hdr.fmt == Q2_NOWEIGHTS) return Q2_EFMT;
  return q2_launch_decode(h, out_dev, static_cast<void*>(stream));
}

}  // extern "C"
