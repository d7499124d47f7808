// Host side of the fused decode step: ring geometry, and the dispatch to
// the instantiations compiled in decode_fused_{bf16,bf16_u8,f32}.cu.
#include "decode_fused.cuh"

namespace q3 {

using namespace fused;

int fused_decode_nq_max() { return FD_NQ; }
int fused_decode_chunk() { return FD_ITEM; }

// Ring geometry for this model: slot = the largest weight row (gate|up pair)
// of a unit, at least 16 KB; union area = the staged inputs of the widest
// phase, or the attention scratch; the rest of shared memory is ring.
bool fused_decode_plan(int dt, int wfmt, FusedArgs& a, size_t* smem) {
  const int esz = dt == DT_BF16 ? 2 : 4, wbytes = wfmt == W_U8 ? 1 : esz;
  if (a.T < 1 || a.T > 4 || a.D != 128 || a.KV < 1 || a.H % a.KV || a.H / a.KV > FD_NQ) return false;
  if (dt != DT_BF16 && wfmt == W_U8) return false;
  const int kmax = std::max(a.hidden, std::max(a.H * a.D, a.I));
  const int rb_max = std::max(2 * a.hidden * wbytes, std::max(a.H * a.D * wbytes, a.I * wbytes));
  const int kv_unit = 2 * FD_KW * a.D * esz;
  int slot = 16 * 1024;
  while (slot < rb_max || slot < kv_unit) slot += 1024;
  a.slot_bytes = slot;
  a.u_bytes = (int)fd_align((size_t)a.T * kmax * esz, 128);
  const size_t limit = 227 * 1024 - 512;  // leave room for the kernel's static shared memory
  a.n_slots = 0;
  for (int ns = 64; ns >= 4; --ns) {
    a.n_slots = ns;
    if (fd_geom(a, FDL<128>::ATT_BYTES).total <= limit) break;
    a.n_slots = 0;
  }
  if (a.n_slots == 0) return false;
  *smem = fd_geom(a, FDL<128>::ATT_BYTES).total;
  return true;
}

cudaError_t launch_fused_decode(const LaunchCtx& c, int dt, int wfmt, const FusedArgs& a, int grid, size_t smem) {
  const int nq = a.T * (a.H / a.KV);
  if (dt == DT_BF16) return wfmt == W_U8 ? fused_launch_bf16_u8(c, a, grid, smem, nq) : fused_launch_bf16(c, a, grid, smem, nq);
  return fused_launch_f32(c, a, grid, smem, nq);
}

}  // namespace q3
